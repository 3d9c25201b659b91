"""CPU-only checks of the C-ABI library: it loads, exports every declared
symbol, and its host-side batch planning (validation, positions, slots) is
bit-exact against the oracle's slot function and brute force."""
import ctypes
import os
import re

import numpy as np
import pytest

from chunked_prefill_hybrid_gb300 import native, synth
from oracle import oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build_library()
    return native.lib()


def declared_symbols():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(hb_\w+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert names, "no declarations found"
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(native.ABI_SYMBOLS) <= set(names)


def _cfg(num_blocks=64, max_tokens=512, max_decodes=32, max_pos=1024):
    return native.model_config(synth.TINY, num_blocks, max_tokens, max_decodes, max_pos)


def test_plan_positions_and_slots_bit_exact(L):
    b = synth.hybrid_batch(5, (1,), 37, 29, [0, 15, 16, 100], 64)
    pos, slot = native.plan(_cfg(), native.Spec(b))
    exp_pos = list(range(37, 37 + 29)) + [0, 15, 16, 100]
    assert list(pos) == exp_pos
    seqs = [b.chunk] * 29 + b.decodes
    for r, (p, s) in enumerate(zip(pos, slot)):
        tab = seqs[r].block_table
        assert s == orc.slot(tab, int(p), 64)
        walk = [blk * 16 + o for blk in tab for o in range(16)]
        assert s == walk[p]


def _spec_raw(**kw):
    b = synth.hybrid_batch(6, (1,), 10, 8, [5, 9], 64)
    s = native.Spec(b)
    for k, v in kw.items():
        setattr(s.c, k, v)
    return s


@pytest.mark.parametrize("field,value,code", [
    ("chunk_len", 0, native.HB_EINVAL),            # chunk id set but no rows
    ("chunk_offset", -1, native.HB_EINVAL),
    ("chunk_n_blocks", 1, native.HB_ERANGE),       # table too short for offset + len
    ("n_decodes", 40, native.HB_ERANGE),           # above max_decodes
    ("chunk_req_id", -5, native.HB_EINVAL),
])
def test_plan_rejects(L, field, value, code):
    s = _spec_raw(**{field: value})
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(), s)
    assert e.value.code == code


def test_plan_rejects_bad_block_and_duplicates(L):
    b = synth.hybrid_batch(7, (1,), 10, 8, [5, 9], 64)
    b.decodes[0].block_table[0] = 64  # block id == num_blocks
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(), native.Spec(b))
    assert e.value.code == native.HB_ERANGE
    b = synth.hybrid_batch(7, (1,), 10, 8, [5, 9], 64)
    b.decodes[1].req_id = b.decodes[0].req_id
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(), native.Spec(b))
    assert e.value.code == native.HB_EINVAL
    b = synth.hybrid_batch(7, (1,), 10, 8, [5, 9], 64)
    b.decodes[0].req_id = b.chunk.req_id
    with pytest.raises(native.HbError):
        native.plan(_cfg(), native.Spec(b))
    # two rows writing one slot (overlapping tables)
    b = synth.hybrid_batch(7, (1,), 10, 8, [5, 5], 64)
    b.decodes[1].block_table = b.decodes[0].block_table.copy()
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(), native.Spec(b))
    assert e.value.code == native.HB_EINVAL


def test_plan_limits(L):
    # max_tokens exactly reached is fine, one more is not
    b = synth.hybrid_batch(8, (1,), 0, 30, [3, 4], 64)
    assert len(native.plan(_cfg(max_tokens=32), native.Spec(b))[0]) == 32
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(max_tokens=31), native.Spec(b))
    assert e.value.code == native.HB_ERANGE
    # position == max_pos is rejected
    b = synth.hybrid_batch(8, (1,), None, 0, [1023], 80)
    native.plan(_cfg(num_blocks=80, max_pos=1024), native.Spec(b))
    b = synth.hybrid_batch(8, (1,), None, 0, [1024], 80)
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(num_blocks=80, max_pos=1024), native.Spec(b))
    assert e.value.code == native.HB_ERANGE
    # an empty batch
    b = synth.HybridBatch(None, 0, [])
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(), native.Spec(b))
    assert e.value.code == native.HB_EINVAL


def test_decode_only_and_prefill_only_plans(L):
    b = synth.hybrid_batch(9, (1,), None, 0, [0, 1, 31, 32], 64)
    pos, slot = native.plan(_cfg(), native.Spec(b))
    assert list(pos) == [0, 1, 31, 32]
    b = synth.hybrid_batch(9, (1,), 0, 100, [], 64)
    pos, slot = native.plan(_cfg(), native.Spec(b))
    assert list(pos) == list(range(100))
    assert len(set(slot.tolist())) == 100


def _multi(seed=10, n_more=2, nb=96):
    """First chunk 8 @ 10, further chunks (5 @ 0, 12 @ 30, ...) and decodes at 5 and 9."""
    more_shapes = [(0, 5), (30, 12), (3, 1)][:n_more] + [(0, 2)] * max(0, n_more - 3)
    lengths = [18, 6, 10] + [o + n for o, n in more_shapes]
    tabs = synth.allocate_tables(seed, (1,), lengths, nb)
    b = synth.HybridBatch(synth.Seq(0, 10, tabs[0]), 8, [synth.Seq(1, 5, tabs[1]), synth.Seq(2, 9, tabs[2])],
                          [(synth.Seq(10 + i, o, tabs[3 + i]), n) for i, (o, n) in enumerate(more_shapes)])
    return b


def test_plan_several_chunks_rows_and_slots(L):
    b = _multi()
    pos, slot = native.plan(_cfg(num_blocks=96), native.Spec(b))
    assert b.n_tokens == 8 + 5 + 12 + 2
    exp = list(range(10, 18)) + list(range(0, 5)) + list(range(30, 42)) + [5, 9]
    assert list(pos) == exp
    seqs = [b.chunk] * 8 + [b.more_chunks[0][0]] * 5 + [b.more_chunks[1][0]] * 12 + b.decodes
    for r, (p, s) in enumerate(zip(pos, slot)):
        assert s == orc.slot(seqs[r].block_table, int(p), 96)


def test_plan_several_chunks_rejects(L):
    cfg = _cfg(num_blocks=96)
    # HB_MAX_CHUNKS chunks are fine, one more is not
    tabs = synth.allocate_tables(11, (1,), [2] * 17, 96)
    b = synth.HybridBatch(synth.Seq(0, 0, tabs[0]), 2, [],
                          [(synth.Seq(1 + i, 0, tabs[1 + i]), 2) for i in range(native.HB_MAX_CHUNKS - 1)])
    assert len(native.plan(cfg, native.Spec(b))[0]) == 2 * native.HB_MAX_CHUNKS
    b.more_chunks.append((synth.Seq(99, 0, tabs[16]), 2))
    with pytest.raises(native.HbError) as e:
        native.plan(cfg, native.Spec(b))
    assert e.value.code == native.HB_ERANGE
    # further chunks without a first chunk
    b = _multi()
    s = native.Spec(b)
    s.c.chunk_req_id, s.c.chunk_len = -1, 0
    with pytest.raises(native.HbError) as e:
        native.plan(cfg, s)
    assert e.value.code == native.HB_EINVAL
    # a further chunk of length 0, a duplicate id, overlapping tables, a short table
    for how, code in (("len0", native.HB_EINVAL), ("dup", native.HB_EINVAL), ("overlap", native.HB_EINVAL),
                      ("short", native.HB_ERANGE), ("neg", native.HB_EINVAL)):
        b = _multi()
        seq, n = b.more_chunks[1]
        if how == "len0":
            b.more_chunks[1] = (seq, 0)
        elif how == "dup":
            seq.req_id = b.decodes[0].req_id
        elif how == "overlap":
            seq.block_table = b.chunk.block_table.copy()
            seq.cached, b.more_chunks[1] = 10, (seq, 8)
        elif how == "short":
            b.more_chunks[1] = (seq, n + 16)
        else:
            seq.cached = -1
        with pytest.raises(native.HbError) as e:
            native.plan(cfg, native.Spec(b))
        assert e.value.code == code, how
    # rows of all chunks count against max_tokens
    with pytest.raises(native.HbError) as e:
        native.plan(_cfg(num_blocks=96, max_tokens=26), native.Spec(_multi()))
    assert e.value.code == native.HB_ERANGE
