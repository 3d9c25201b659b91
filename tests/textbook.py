"""A textbook LLaMA decoder layer in fp64 PyTorch CPU ops, for pinning the oracle.

It is written with library routines (``F.rms_norm``, ``F.linear``,
``F.scaled_dot_product_attention``, ``F.silu``) and a complex-number form of
rotary embedding, over one dense, unpaged, unchunked sequence starting at
position 0 -- the "full prefill" that chunked prefill is stated to equal
(SARATHI summary, section 3.4 "Chunked-Prefills", Figure 6).  It shares no
code with the oracle.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _w(bits) -> torch.Tensor:
    b = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).astype(np.int32) << 16)
    return b.view(torch.float32).to(torch.float64)


def rope_complex(x: torch.Tensor, positions: torch.Tensor, theta: float) -> torch.Tensor:
    """x: [n][heads][d]; pair (j, j + d/2) as a complex number times e^{i pos theta^(-2j/d)}."""
    d = x.shape[-1]
    half = d // 2
    freqs = theta ** (-torch.arange(0, half, dtype=torch.float64) * 2.0 / d)
    ang = positions.to(torch.float64)[:, None] * freqs[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def layer_full_sequence(dims, weights: dict, x: np.ndarray, gqa_repeat: bool = True):
    """y, plus (q, k, v, o) of one sequence at positions 0..n-1, fp64."""
    X = torch.from_numpy(np.asarray(x, np.float64))
    n, H = X.shape
    nh, nkv, d, Fd = dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.ffn
    wqkv = _w(weights["w_qkv"])
    wq, wk, wv = wqkv[:nh * d], wqkv[nh * d:(nh + nkv) * d], wqkv[(nh + nkv) * d:]
    g1, g2 = _w(weights["norm1"]), _w(weights["norm2"])
    pos = torch.arange(n)
    n1 = F.rms_norm(X, (H,), weight=g1, eps=dims.rms_eps)
    q = rope_complex(F.linear(n1, wq).view(n, nh, d), pos, dims.rope_theta)
    k = rope_complex(F.linear(n1, wk).view(n, nkv, d), pos, dims.rope_theta)
    v = F.linear(n1, wv).view(n, nkv, d)
    kk, vv = k, v
    if nkv != nh and gqa_repeat:
        kk = k.repeat_interleave(nh // nkv, dim=1)
        vv = v.repeat_interleave(nh // nkv, dim=1)
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], kk.transpose(0, 1)[None],
                                       vv.transpose(0, 1)[None], is_causal=True)
    o = o[0].transpose(0, 1).reshape(n, nh * d)
    h = X + F.linear(o, _w(weights["w_o"]))
    n2 = F.rms_norm(h, (H,), weight=g2, eps=dims.rms_eps)
    gu = F.linear(n2, _w(weights["w_gate_up"]))
    a = F.silu(gu[:, :Fd]) * gu[:, Fd:]
    y = h + F.linear(a, _w(weights["w_down"]))
    return (y.numpy(), q.reshape(n, nh * d).numpy(), k.reshape(n, nkv * d).numpy(),
            v.reshape(n, nkv * d).numpy(), o.numpy())
