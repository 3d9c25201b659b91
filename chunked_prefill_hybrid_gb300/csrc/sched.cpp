// sched.cpp -- the host decode-maximal scheduler behind include/hb_sched.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <map>
#include <set>
#include <vector>

#include "hb_sched.h"

namespace {

enum Phase { WAITING = 0, PREFILL = 1, DECODE = 2, DONE = 3 };

struct Req {
    int id = 0, prompt = 0, max_new = 0;
    int processed = 0;   // prompt tokens in the KV cache
    int generated = 0;   // tokens produced so far
    Phase phase = WAITING;
    long long order = 0; // admission order
    std::vector<int32_t> blocks;
};

}  // namespace

struct hb_sched {
    hb_sched_config cfg{};
    std::map<int, Req> reqs;
    std::deque<int> waiting;            // FCFS
    std::vector<int> running;           // admitted, in admission order
    std::set<int32_t> free_blocks;      // lowest id first
    long long admit_counter = 0;
    // last batch
    std::vector<int32_t> c_ids, c_off, c_len, d_ids, d_ctx;
    int n_rows = 0;
    bool pending = false;
    std::vector<int32_t> spec_dbt, spec_mbt, spec_mids;
    hb_sched_stats stats{};
    double pd_ewma = -1.0;  // P:D of finished requests, exponentially weighted
};

static constexpr double kPdWeight = 0.125;  // weight of the newest observation

static int blocks_for(const hb_sched_config &c, long long tokens)
{
    return (int)((tokens + c.block_size - 1) / c.block_size);
}

extern "C" int hb_sched_create(const hb_sched_config *cfg, hb_sched **out)
{
    if (!out)
        return HB_EINVAL;
    *out = nullptr;
    if (!cfg || cfg->chunk_size <= 0 || cfg->max_decodes < 0 || cfg->tile < 0 || cfg->max_chunks_per_batch < 1 ||
        cfg->block_size <= 0 || cfg->num_blocks < 0 || cfg->max_blocks_per_seq <= 0 || cfg->request_level < 0 ||
        cfg->request_level > 1)
        return HB_EINVAL;
    hb_sched *s = new hb_sched();
    s->cfg = *cfg;
    for (int b = 0; b < cfg->num_blocks; ++b)
        s->free_blocks.insert(b);
    *out = s;
    return HB_OK;
}

extern "C" int hb_sched_add(hb_sched *s, int req_id, int prompt_len, int max_new_tokens)
{
    if (!s || req_id < 0 || prompt_len < 1 || max_new_tokens < 1)
        return HB_EINVAL;
    if (s->reqs.count(req_id))
        return HB_EINVAL;
    const int need = blocks_for(s->cfg, (long long)prompt_len + max_new_tokens);
    if (need > s->cfg.num_blocks || need > s->cfg.max_blocks_per_seq)
        return HB_ENOMEM;
    Req r;
    r.id = req_id;
    r.prompt = prompt_len;
    r.max_new = max_new_tokens;
    s->reqs[req_id] = r;
    s->waiting.push_back(req_id);
    return HB_OK;
}

static void admit(hb_sched *s)
{
    const bool request_level = s->cfg.request_level != 0;
    if (request_level && !s->running.empty())
        return;  // a request-level batch forms only when the previous one has finished
    const size_t cap = request_level ? (size_t)std::max(1, s->cfg.max_decodes) : (size_t)-1;
    while (!s->waiting.empty() && s->running.size() < cap) {
        Req &r = s->reqs[s->waiting.front()];
        const int need = blocks_for(s->cfg, (long long)r.prompt + r.max_new);
        if ((int)s->free_blocks.size() < need)
            break;  // first come first served: no overtaking
        for (int i = 0; i < need; ++i) {
            r.blocks.push_back(*s->free_blocks.begin());
            s->free_blocks.erase(s->free_blocks.begin());
        }
        r.phase = PREFILL;
        r.order = s->admit_counter++;
        s->running.push_back(r.id);
        s->waiting.pop_front();
    }
}

extern "C" int hb_sched_next(hb_sched *s, hb_sched_batch *out)
{
    if (!s || !out)
        return HB_EINVAL;
    if (s->pending)
        return HB_ESTATE;  // hb_sched_complete first
    admit(s);
    const hb_sched_config &c = s->cfg;
    const long long budget = c.token_budget > 0 ? c.token_budget : (1ll << 40);
    s->c_ids.clear();
    s->c_off.clear();
    s->c_len.clear();
    s->d_ids.clear();
    s->d_ctx.clear();
    long long rows = 0;
    bool prefill_left = false;
    for (int id : s->running)
        prefill_left = prefill_left || s->reqs[id].phase == PREFILL;
    const bool take_decodes = !c.request_level || !prefill_left;
    // decodes first, admission order
    for (int id : s->running) {
        if (!take_decodes)
            break;
        const Req &r = s->reqs[id];
        if (r.phase != DECODE)
            continue;
        if ((int)s->d_ids.size() >= c.max_decodes || rows + 1 > budget)
            break;
        s->d_ids.push_back(id);
        s->d_ctx.push_back(r.prompt + r.generated - 1);
        rows += 1;
    }
    // then chunks, oldest admitted request with prompt left first
    for (int id : s->running) {
        if ((int)s->c_ids.size() >= c.max_chunks_per_batch || rows >= budget)
            break;
        const Req &r = s->reqs[id];
        if (r.phase != PREFILL)
            continue;
        long long len = std::min<long long>(c.chunk_size, r.prompt - r.processed);
        len = std::min(len, budget - rows);
        if (len <= 0)
            break;
        s->c_ids.push_back(id);
        s->c_off.push_back(r.processed);
        s->c_len.push_back((int32_t)len);
        rows += len;
    }
    if (c.tile > 0 && s->c_ids.size() == 1) {
        const long long rem = rows % c.tile;
        if (rem != 0 && s->c_len[0] > rem) {
            s->c_len[0] -= (int32_t)rem;
            rows -= rem;
        }
    }
    s->n_rows = (int)rows;
    out->n_chunks = (int)s->c_ids.size();
    out->chunk_req_ids = s->c_ids.data();
    out->chunk_offsets = s->c_off.data();
    out->chunk_lens = s->c_len.data();
    out->n_decodes = (int)s->d_ids.size();
    out->decode_req_ids = s->d_ids.data();
    out->decode_ctx_lens = s->d_ctx.data();
    out->n_rows = s->n_rows;
    s->pending = rows > 0;
    if (rows > 0) {
        s->stats.iterations++;
        s->stats.rows += rows;
        if (s->c_ids.empty())
            s->stats.decode_only_iterations++;
    }
    return (int)rows;
}

extern "C" int hb_sched_complete(hb_sched *s)
{
    if (!s)
        return HB_EINVAL;
    if (!s->pending)
        return HB_ESTATE;
    s->pending = false;
    int finished = 0;
    auto finish = [&](Req &r) {
        const double pd = (double)r.prompt / (double)r.generated;
        s->pd_ewma = s->pd_ewma < 0 ? pd : s->pd_ewma + kPdWeight * (pd - s->pd_ewma);
        r.phase = DONE;
        for (int32_t b : r.blocks)
            s->free_blocks.insert(b);
        r.blocks.clear();
        s->running.erase(std::find(s->running.begin(), s->running.end(), r.id));
        ++finished;
    };
    for (size_t i = 0; i < s->c_ids.size(); ++i) {
        Req &r = s->reqs[s->c_ids[i]];
        r.processed += s->c_len[i];
        if (r.processed == r.prompt) {
            r.generated = 1;  // the last prompt chunk yields the first token
            if (r.generated >= r.max_new)
                finish(r);
            else
                r.phase = DECODE;
        }
    }
    for (int32_t id : s->d_ids) {
        Req &r = s->reqs[id];
        r.generated += 1;
        if (r.generated >= r.max_new)
            finish(r);
    }
    return finished;
}

extern "C" int hb_sched_block_table(hb_sched *s, int req_id, const int32_t **table, int *n_blocks)
{
    if (!s || !table || !n_blocks)
        return HB_EINVAL;
    auto it = s->reqs.find(req_id);
    if (it == s->reqs.end() || it->second.blocks.empty())
        return HB_EINVAL;
    *table = it->second.blocks.data();
    *n_blocks = (int)it->second.blocks.size();
    return HB_OK;
}

extern "C" int hb_sched_fill_spec(hb_sched *s, hb_batch_spec *spec)
{
    if (!s || !spec)
        return HB_EINVAL;
    if (s->c_ids.size() > HB_MAX_CHUNKS)
        return HB_ERANGE;
    std::memset(spec, 0, sizeof *spec);
    spec->chunk_req_id = -1;
    if (!s->c_ids.empty()) {
        const Req &r = s->reqs[s->c_ids[0]];
        spec->chunk_req_id = r.id;
        spec->chunk_offset = s->c_off[0];
        spec->chunk_len = s->c_len[0];
        spec->chunk_block_table = r.blocks.data();
        spec->chunk_n_blocks = (int)r.blocks.size();
    }
    const int W = s->cfg.max_blocks_per_seq;
    const size_t n_more = s->c_ids.empty() ? 0 : s->c_ids.size() - 1;
    s->spec_mbt.assign(std::max<size_t>(1, n_more) * W, -1);
    s->spec_mids.assign(std::max<size_t>(1, n_more), 0);
    for (size_t i = 0; i < n_more; ++i) {
        const Req &r = s->reqs[s->c_ids[i + 1]];
        s->spec_mids[i] = r.id;
        std::copy(r.blocks.begin(), r.blocks.end(), s->spec_mbt.begin() + i * W);
    }
    spec->n_more_chunks = (int)n_more;
    spec->more_chunk_req_ids = s->spec_mids.data();
    spec->more_chunk_offsets = s->c_off.data() + (n_more ? 1 : 0);
    spec->more_chunk_lens = s->c_len.data() + (n_more ? 1 : 0);
    spec->more_chunk_block_tables = s->spec_mbt.data();
    spec->more_chunk_bt_stride = W;
    s->spec_dbt.assign((size_t)std::max<size_t>(1, s->d_ids.size()) * W, -1);
    for (size_t j = 0; j < s->d_ids.size(); ++j) {
        const Req &r = s->reqs[s->d_ids[j]];
        std::copy(r.blocks.begin(), r.blocks.end(), s->spec_dbt.begin() + j * W);
    }
    spec->n_decodes = (int)s->d_ids.size();
    spec->decode_req_ids = s->d_ids.data();
    spec->decode_ctx_lens = s->d_ctx.data();
    spec->decode_block_tables = s->spec_dbt.data();
    spec->decode_bt_stride = W;
    return HB_OK;
}

extern "C" int hb_sched_get_stats(hb_sched *s, hb_sched_stats *out)
{
    if (!s || !out)
        return HB_EINVAL;
    hb_sched_stats st = s->stats;
    st.waiting = (int)s->waiting.size();
    st.prefilling = st.decoding = st.finished = 0;
    for (auto &kv : s->reqs) {
        if (kv.second.phase == PREFILL)
            st.prefilling++;
        else if (kv.second.phase == DECODE)
            st.decoding++;
        else if (kv.second.phase == DONE)
            st.finished++;
    }
    st.free_blocks = (int)s->free_blocks.size();
    *out = st;
    return HB_OK;
}

extern "C" long long hb_sched_max_batch(long long mem_total, long long mem_params, long long max_len,
                                        long long kv_bytes_per_token)
{
    if (mem_total <= 0 || mem_params < 0 || max_len <= 0 || kv_bytes_per_token <= 0 || mem_total <= mem_params)
        return -1;
    return (mem_total - mem_params) / (max_len * kv_bytes_per_token);
}

extern "C" void hb_sched_free(hb_sched *s) { delete s; }

extern "C" double hb_perfect_pd_ratio(int chunk_size, int batch_size)
{
    if (chunk_size < 1 || batch_size < 2)
        return -1.0;
    return (double)chunk_size / (double)(batch_size - 1);
}

extern "C" long long hb_piggyback_capacity(long long prompt_len, long long decode_len, int chunk_size, int batch_size)
{
    if (prompt_len < 1 || decode_len < 0 || chunk_size < 1 || batch_size < 1)
        return -1;
    const long long chunks = (prompt_len + chunk_size - 1) / chunk_size;
    const long long cap = chunks * (long long)(batch_size - 1);
    return decode_len < cap ? decode_len : cap;
}

extern "C" int hb_advise_chunk(double pd_ratio, int batch_size, int tile, int c_min, int c_max)
{
    if (!(pd_ratio > 0) || batch_size < 2 || c_min < 1 || c_max < c_min || tile < 0)
        return -1;
    const double want = pd_ratio * (double)(batch_size - 1);
    long long c0 = (long long)std::llround(want);
    if (c0 < c_min)
        c0 = c_min;
    if (c0 > c_max)
        c0 = c_max;
    if (tile == 0)
        return (int)c0;
    const long long rows = c0 + batch_size - 1;
    const long long c = rows / tile * tile - (batch_size - 1);
    return (int)(c >= c_min ? c : c0);
}

extern "C" double hb_sched_pd_estimate(hb_sched *s) { return s ? s->pd_ewma : -1.0; }
