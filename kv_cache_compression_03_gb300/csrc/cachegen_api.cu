// Host side of the CacheGen codec's C ABI: configuration checks, the plan
// (tile table, buffer sizes, workspace layout), kernel launches, and the
// flat container. The operations are defined in include/cachegen.h.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "cg_internal.h"

namespace {

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Expand spec triples into one bin count per layer: [start, end) ranges that
// cover [0, L) exactly once, bins even in [4, 64] ("LMCache 中的 KV Cache 压缩：
// CacheGen 编解码原理、配置方式与源码解析", §1 QuantizationSpec).
cg_status expand_specs(int32_t L, const cg_quant_spec *specs, int32_t n, uint8_t *bins)
{
    if (specs == nullptr || n <= 0)
        return CG_ERR_INVALID_ARG;
    for (int32_t l = 0; l < L; ++l)
        bins[l] = 0;
    for (int32_t i = 0; i < n; ++i) {
        const cg_quant_spec &s = specs[i];
        if (s.start_layer < 0 || s.end_layer > L || s.start_layer >= s.end_layer)
            return CG_ERR_SPEC;
        if (s.bins < 4 || s.bins > 64 || (s.bins & 1))
            return CG_ERR_SPEC;
        for (int32_t l = s.start_layer; l < s.end_layer; ++l) {
            if (bins[l] != 0)
                return CG_ERR_SPEC;
            bins[l] = (uint8_t)s.bins;
        }
    }
    for (int32_t l = 0; l < L; ++l)
        if (bins[l] == 0)
            return CG_ERR_SPEC;
    return CG_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr uint32_t kMagic = 0x564B4743u;  // "CGKV" little-endian
constexpr uint32_t kVersion = 1;
constexpr size_t kHeaderFixed = 48;

void put32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }  // hosts are little-endian
uint32_t get32(const uint8_t *p)
{
    uint32_t v;
    memcpy(&v, p, 4);
    return v;
}

size_t header_bytes(const cg_plan *p)
{
    return kHeaderFixed + 12 * (p->kspecs.size() + p->vspecs.size());
}

struct Sections {
    size_t amax, lengths, cdf, streams, end;
};

// Section offsets of a container holding T tokens in ngroups groups.
Sections sections_for(const cg_plan *p, int64_t T, int64_t ngroups, uint64_t stream_bytes)
{
    const size_t streams = (size_t)2 * p->L * (size_t)T;
    Sections s;
    s.amax = header_bytes(p);
    s.lengths = s.amax + 4 * streams;
    s.cdf = s.lengths + 4 * streams;
    s.streams = s.cdf + 2 * (size_t)p->tp.cdf_per_group * (size_t)ngroups;
    s.end = s.streams + (size_t)stream_bytes;
    return s;
}

Sections sections(const cg_plan *p, uint64_t stream_bytes)
{
    return sections_for(p, p->T, p->tp.ngroups, stream_bytes);
}

// Header and spec lists of a container of T tokens in ngroups groups.
void write_header(uint8_t *h, const cg_plan *p, int32_t T, int32_t ngroups, uint64_t stream_bytes)
{
    put32(h + 0, kMagic);
    put32(h + 4, kVersion);
    put32(h + 8, (uint32_t)p->L);
    put32(h + 12, (uint32_t)T);
    put32(h + 16, (uint32_t)p->H);
    put32(h + 20, (uint32_t)p->D);
    put32(h + 24, (uint32_t)p->chunk_tokens);
    put32(h + 28, (uint32_t)p->kspecs.size());
    put32(h + 32, (uint32_t)p->vspecs.size());
    put32(h + 36, (uint32_t)ngroups);
    put32(h + 40, (uint32_t)(stream_bytes & 0xFFFFFFFFu));
    put32(h + 44, (uint32_t)(stream_bytes >> 32));
    uint8_t *q = h + kHeaderFixed;
    for (const auto *list : {&p->kspecs, &p->vspecs})
        for (const cg_quant_spec &s : *list) {
            put32(q, (uint32_t)s.start_layer);
            put32(q + 4, (uint32_t)s.end_layer);
            put32(q + 8, (uint32_t)s.bins);
            q += 12;
        }
}

// Objects: runs of chunk_tokens tokens (the last may be shorter); groups
// never span two objects, so object o owns groups [g0, g0 + ng).
struct ObjectRange {
    int32_t t0, n, g0, ng;
};

int32_t num_objects(const cg_plan *p)
{
    return p->tp.full_objects + ((int64_t)p->tp.full_objects * p->chunk_tokens < p->T ? 1 : 0);
}

bool object_range(const cg_plan *p, int32_t o, ObjectRange *r)
{
    if (o < 0 || o >= num_objects(p))
        return false;
    const int64_t t0 = (int64_t)o * p->chunk_tokens;
    const int64_t n = std::min<int64_t>(p->chunk_tokens, p->T - t0);
    r->t0 = (int32_t)t0;
    r->n = (int32_t)n;
    r->g0 = o * p->tp.groups_per_object;
    r->ng = (int32_t)((n + CG_GROUP_TOKENS - 1) / CG_GROUP_TOKENS);
    return true;
}

}  // namespace

extern "C" {

const char *cg_status_string(cg_status st)
{
    switch (st) {
    case CG_OK: return "ok";
    case CG_ERR_INVALID_ARG: return "invalid argument";
    case CG_ERR_SPEC: return "invalid quantisation spec";
    case CG_ERR_CAPACITY: return "output capacity exceeded";
    case CG_ERR_NONFINITE: return "non-finite input";
    case CG_ERR_CORRUPT: return "corrupt container";
    case CG_ERR_TIMEOUT: return "device wait timed out";
    case CG_ERR_CUDA: return "CUDA error";
    case CG_ERR_UNSUPPORTED: return "shape not supported";
    }
    return "unknown status";
}

cg_status cg_plan_create(const cg_config *cfg, cg_plan **plan_out)
{
    if (cfg == nullptr || plan_out == nullptr)
        return CG_ERR_INVALID_ARG;
    *plan_out = nullptr;
    const int32_t L = cfg->num_layers, T = cfg->num_tokens;
    const int32_t H = cfg->num_heads, D = cfg->head_size, ch = cfg->chunk_tokens;
    if (L <= 0 || T <= 0 || H <= 0 || D <= 0 || ch <= 0)
        return CG_ERR_INVALID_ARG;
    if ((int64_t)H * D > CG_MAX_CHANNELS || L > CG_MAX_LAYERS)
        return CG_ERR_UNSUPPORTED;
    const int32_t C = H * D;
    if (C % 8 != 0)
        return CG_ERR_INVALID_ARG;
    cg_plan *p = new (std::nothrow) cg_plan();
    if (!p)
        return CG_ERR_INVALID_ARG;
    p->L = L;
    p->T = T;
    p->H = H;
    p->D = D;
    p->C = C;
    p->chunk_tokens = ch;
    memset(&p->tp, 0, sizeof p->tp);
    cg_status st = expand_specs(L, cfg->kspecs, cfg->n_kspecs, p->tp.bins[0]);
    if (st == CG_OK)
        st = expand_specs(L, cfg->vspecs, cfg->n_vspecs, p->tp.bins[1]);
    if (st != CG_OK) {
        delete p;
        return st;
    }
    p->kspecs.assign(cfg->kspecs, cfg->kspecs + cfg->n_kspecs);
    p->vspecs.assign(cfg->vspecs, cfg->vspecs + cfg->n_vspecs);

    // token groups: objects of ch tokens, each cut into groups of <= 256
    cg_tile_params &tp = p->tp;
    tp.L = L;
    tp.T = T;
    tp.C = C;
    tp.chunk_tokens = ch;
    tp.one = 1;
    tp.groups_per_object = (ch + CG_GROUP_TOKENS - 1) / CG_GROUP_TOKENS;
    tp.full_objects = T / ch;
    const int32_t tail = T - tp.full_objects * ch;
    const int64_t ngroups =
        (int64_t)tp.full_objects * tp.groups_per_object + (tail + CG_GROUP_TOKENS - 1) / CG_GROUP_TOKENS;
    const int64_t ntiles = ngroups * 2 * L;
    if (ntiles > (int64_t)INT32_MAX / 2) {
        delete p;
        return CG_ERR_UNSUPPORTED;
    }
    tp.ngroups = (int32_t)ngroups;
    tp.ntiles = (int32_t)ntiles;

    // CDF block offsets: per group, K/V, layer, channel, N+1 entries
    uint64_t off = 0;
    int32_t maxb = 0;
    for (int kv = 0; kv < 2; ++kv)
        for (int32_t l = 0; l < L; ++l) {
            tp.cdf_off[kv][l] = (uint32_t)off;
            off += (uint64_t)C * (tp.bins[kv][l] + 1);
            if (tp.bins[kv][l] > maxb)
                maxb = tp.bins[kv][l];
        }
    tp.cdf_per_group = off;
    p->max_bins = maxb;
    p->cdf_entries = off * (uint64_t)ngroups;
    p->num_streams = (uint64_t)2 * L * T;

    // a stream of C symbols needs at most C + 1 bytes when every coded
    // symbol has frequency >= 256 of 2^16 (true for groups of <= 256
    // tokens: a symbol that occurs has count >= 1); a slot is a 16-byte pad
    // (the encoder may write the word before a stream's first one there)
    // and then room for C + 16 bytes
    tp.slot_stride = (uint32_t)align_up((size_t)C + 32, 16);
    p->max_stream_bytes = align_up((size_t)p->num_streams * (C + 2), 16);

    // tile order: (kv, layer) pairs by bin count, largest first
    {
        int32_t k = 0;
        p->smem_encode = p->smem_decode = 0;
        for (int32_t b = 64; b >= 4; b -= 2) {
            for (int kv = 0; kv < 2; ++kv)
                for (int32_t l = 0; l < L; ++l)
                    if (tp.bins[kv][l] == b)
                        tp.order[k++] = (uint16_t)((kv << 8) | l);
        }
        p->smem_encode = cg_smem_encode(C, maxb);
        p->smem_decode = cg_smem_decode(C, maxb);
        for (int32_t i = 0; i < k;) {
            cg_bin_class cl;
            cl.begin = i;
            cl.bins = tp.bins[tp.order[i] >> 8][tp.order[i] & 0xFF];
            while (i < k && tp.bins[tp.order[i] >> 8][tp.order[i] & 0xFF] == cl.bins)
                ++i;
            cl.count = i - cl.begin;
            cl.smem_encode = cg_smem_encode(C, cl.bins);
            cl.smem_decode = cg_smem_decode(C, cl.bins);
            p->classes.push_back(cl);
        }
        if (p->smem_encode > CG_SMEM_LIMIT - 2048 || p->smem_decode > CG_SMEM_LIMIT - 2048) {
            delete p;
            return CG_ERR_UNSUPPORTED;
        }
        // 16-bin symbols (at most 14) as 4-bit codes when the encoder's
        // four-channels-per-thread path runs and rows stay 16-byte aligned
        tp.nib_begin = tp.nib_end = 0;
        int32_t w16 = 0, r16 = 0;
        cg_count_layout(C, 16, &w16, &r16);
        if (w16 == 4 && C % 32 == 0)
            for (const cg_bin_class &cl : p->classes)
                if (cl.bins == 16) {
                    tp.nib_begin = cl.begin;
                    tp.nib_end = cl.begin + cl.count;
                }
    }

    // workspace: status | tile totals | tile bases | symbols | slots
    size_t w = CG_WS_STATUS_BYTES;
    p->ws_tile_totals = w;
    w = align_up(w + 4 * (size_t)ntiles, 256);
    p->ws_tile_base = w;
    w = align_up(w + 8 * ((size_t)ntiles + 1), 256);
    p->ws_symbols = w;
    const size_t nib_pairs = (size_t)(tp.nib_end - tp.nib_begin);
    w = align_up(w + (size_t)T * ((size_t)C * 2 * L - (size_t)(C / 2) * nib_pairs), 256);
    p->ws_slots = w;
    w = align_up(w + (size_t)p->num_streams * tp.slot_stride, 256);
    p->ws_bytes = w;
    *plan_out = p;
    return CG_OK;
}

void cg_plan_destroy(cg_plan *plan)
{
    if (plan) {
        cg_profile_enable(plan, 0);
        plan->side.release();
    }
    delete plan;
}

cg_status cg_profile_enable(cg_plan *p, int32_t max_launches)
{
    if (p == nullptr || max_launches < 0)
        return CG_ERR_INVALID_ARG;
    for (cudaEvent_t e : p->prof.events)
        cudaEventDestroy(e);
    p->prof.events.clear();
    p->prof.ids.clear();
    p->prof.used = 0;
    if (max_launches == 0)
        return CG_OK;
    p->prof.events.resize((size_t)max_launches * 2, nullptr);
    p->prof.ids.resize((size_t)max_launches, 0);
    for (cudaEvent_t &e : p->prof.events)
        if (cudaEventCreate(&e) != cudaSuccess) {
            p->prof.events.clear();
            return CG_ERR_CUDA;
        }
    return CG_OK;
}

cg_status cg_profile_read(cg_plan *p, cg_kernel_profile *out, int32_t capacity, int32_t *count)
{
    if (p == nullptr || count == nullptr || (capacity > 0 && out == nullptr))
        return CG_ERR_INVALID_ARG;
    double ms[CG_K_COUNT] = {0};
    int64_t n[CG_K_COUNT] = {0};
    for (int32_t i = 0; i < p->prof.used; ++i) {
        float t = 0.0f;
        if (cudaEventSynchronize(p->prof.events[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&t, p->prof.events[2 * i], p->prof.events[2 * i + 1]) !=
                cudaSuccess)
            return CG_ERR_CUDA;
        ms[p->prof.ids[i]] += t;
        n[p->prof.ids[i]] += 1;
    }
    p->prof.used = 0;
    int32_t k = 0;
    for (int id = 0; id < CG_K_COUNT; ++id) {
        if (n[id] == 0)
            continue;
        if (k < capacity) {
            out[k].kernel = cg_kernel_name(id);
            out[k].launches = n[id];
            out[k].total_ms = ms[id];
        }
        ++k;
    }
    *count = k;
    return CG_OK;
}

cg_status cg_plan_sizes(const cg_plan *p, cg_sizes *out)
{
    if (p == nullptr || out == nullptr)
        return CG_ERR_INVALID_ARG;
    out->workspace_bytes = p->ws_bytes;
    out->max_stream_bytes = p->max_stream_bytes;
    out->cdf_entries = (size_t)p->cdf_entries;
    out->num_streams = (size_t)p->num_streams;
    out->num_scales = (size_t)p->num_streams;
    out->raw_bytes = (size_t)p->num_streams * p->C * 2;
    out->num_groups = p->tp.ngroups;
    out->num_tiles = p->tp.ntiles;
    out->encode_launches = cg_encode_launch_count(p);
    out->decode_launches = cg_decode_launch_count(p);
    out->num_objects = num_objects(p);
    return CG_OK;
}

cg_status cg_plan_config(const cg_plan *p, cg_config *out, cg_quant_spec *kspecs, int32_t kcap,
                         cg_quant_spec *vspecs, int32_t vcap)
{
    if (p == nullptr || out == nullptr || kcap < 0 || vcap < 0)
        return CG_ERR_INVALID_ARG;
    if ((kcap > 0 && kspecs == nullptr) || (vcap > 0 && vspecs == nullptr))
        return CG_ERR_INVALID_ARG;
    out->num_layers = p->L;
    out->num_tokens = p->T;
    out->num_heads = p->H;
    out->head_size = p->D;
    out->chunk_tokens = p->chunk_tokens;
    out->n_kspecs = (int32_t)p->kspecs.size();
    out->n_vspecs = (int32_t)p->vspecs.size();
    out->kspecs = kspecs;
    out->vspecs = vspecs;
    if (kcap < out->n_kspecs || vcap < out->n_vspecs)
        return CG_ERR_CAPACITY;
    std::copy(p->kspecs.begin(), p->kspecs.end(), kspecs);
    std::copy(p->vspecs.begin(), p->vspecs.end(), vspecs);
    return CG_OK;
}

cg_status cg_encode(const cg_plan *p, const void *kv, void *workspace, size_t workspace_bytes,
                    const cg_encoded *out, cg_stream_t stream)
{
    if (p == nullptr || kv == nullptr || workspace == nullptr || out == nullptr)
        return CG_ERR_INVALID_ARG;
    if (!out->bytestream || !out->lengths || !out->cdf || !out->amax)
        return CG_ERR_INVALID_ARG;
    if (!aligned(kv, 16) || !aligned(workspace, 256) || !aligned(out->bytestream, 16) ||
        !aligned(out->cdf, 16) || !aligned(out->lengths, 4) || !aligned(out->amax, 4))
        return CG_ERR_INVALID_ARG;
    if (workspace_bytes < p->ws_bytes)
        return CG_ERR_CAPACITY;
    cudaError_t e = cg_launch_encode(p, kv, workspace, out, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}

cg_status cg_decode(const cg_plan *p, const cg_encoded *in, uint64_t stream_bytes, void *workspace,
                    size_t workspace_bytes, void *kv_out, cg_stream_t stream)
{
    if (p == nullptr || in == nullptr || workspace == nullptr || kv_out == nullptr)
        return CG_ERR_INVALID_ARG;
    if (!in->bytestream || !in->lengths || !in->cdf || !in->amax)
        return CG_ERR_INVALID_ARG;
    if (!aligned(kv_out, 16) || !aligned(workspace, 256) || !aligned(in->bytestream, 16) ||
        !aligned(in->cdf, 16) || !aligned(in->lengths, 4) || !aligned(in->amax, 4))
        return CG_ERR_INVALID_ARG;
    if (stream_bytes < p->num_streams)  // every stream has at least one byte
        return CG_ERR_CORRUPT;
    if (in->bytestream_capacity < align_up((size_t)stream_bytes, 16))
        return CG_ERR_CAPACITY;
    // decode needs only the status block, tile totals and tile bases
    if (workspace_bytes < p->ws_symbols)
        return CG_ERR_CAPACITY;
    cudaError_t e = cg_launch_decode(p, in, stream_bytes, workspace, kv_out,
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}

cg_status cg_last_device_error(const cg_plan *p, const void *workspace, cg_status *status,
                               uint64_t *stream_bytes, cg_stream_t stream)
{
    (void)p;  // the status block has the same layout for every plan
    if (workspace == nullptr)
        return CG_ERR_INVALID_ARG;
    uint8_t blk[16];
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(blk, workspace, sizeof blk, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return CG_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return CG_ERR_CUDA;
    uint32_t st;
    uint64_t tot;
    memcpy(&st, blk + CG_WS_STATUS, 4);
    memcpy(&tot, blk + CG_WS_TOTAL, 8);
    if (status)
        *status = (cg_status)st;
    if (stream_bytes)
        *stream_bytes = tot;
    return CG_OK;
}

cg_status cg_container_size(const cg_plan *p, uint64_t stream_bytes, size_t *bytes)
{
    if (p == nullptr || bytes == nullptr)
        return CG_ERR_INVALID_ARG;
    *bytes = sections(p, stream_bytes).end;
    return CG_OK;
}

cg_status cg_serialize(const cg_plan *p, const cg_encoded *enc, uint64_t stream_bytes,
                       void *host_out, size_t host_capacity, size_t *written, cg_stream_t stream)
{
    if (p == nullptr || enc == nullptr || host_out == nullptr)
        return CG_ERR_INVALID_ARG;
    const Sections sec = sections(p, stream_bytes);
    if (host_capacity < sec.end)
        return CG_ERR_CAPACITY;
    if (stream_bytes > enc->bytestream_capacity)
        return CG_ERR_CAPACITY;
    uint8_t *h = static_cast<uint8_t *>(host_out);
    write_header(h, p, p->T, p->tp.ngroups, stream_bytes);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(h + sec.amax, enc->amax, 4 * (size_t)p->num_streams,
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h + sec.lengths, enc->lengths, 4 * (size_t)p->num_streams,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h + sec.cdf, enc->cdf, 2 * (size_t)p->cdf_entries,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && stream_bytes > 0)
        e = cudaMemcpyAsync(h + sec.streams, enc->bytestream, (size_t)stream_bytes,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return CG_ERR_CUDA;
    if (written)
        *written = sec.end;
    return CG_OK;
}

cg_status cg_container_open(const void *host_in, size_t len, cg_plan **plan_out,
                            uint64_t *stream_bytes)
{
    if (host_in == nullptr || plan_out == nullptr)
        return CG_ERR_INVALID_ARG;
    *plan_out = nullptr;
    const uint8_t *h = static_cast<const uint8_t *>(host_in);
    if (len < kHeaderFixed || get32(h) != kMagic || get32(h + 4) != kVersion)
        return CG_ERR_CORRUPT;
    const int32_t nk = (int32_t)get32(h + 28), nv = (int32_t)get32(h + 32);
    if (nk <= 0 || nv <= 0 || nk > CG_MAX_LAYERS || nv > CG_MAX_LAYERS)
        return CG_ERR_CORRUPT;
    if (len < kHeaderFixed + 12 * (size_t)(nk + nv))
        return CG_ERR_CORRUPT;
    std::vector<cg_quant_spec> ks(nk), vs(nv);
    const uint8_t *q = h + kHeaderFixed;
    for (int32_t i = 0; i < nk; ++i, q += 12)
        ks[i] = {(int32_t)get32(q), (int32_t)get32(q + 4), (int32_t)get32(q + 8)};
    for (int32_t i = 0; i < nv; ++i, q += 12)
        vs[i] = {(int32_t)get32(q), (int32_t)get32(q + 4), (int32_t)get32(q + 8)};
    cg_config cfg;
    cfg.num_layers = (int32_t)get32(h + 8);
    cfg.num_tokens = (int32_t)get32(h + 12);
    cfg.num_heads = (int32_t)get32(h + 16);
    cfg.head_size = (int32_t)get32(h + 20);
    cfg.chunk_tokens = (int32_t)get32(h + 24);
    cfg.kspecs = ks.data();
    cfg.n_kspecs = nk;
    cfg.vspecs = vs.data();
    cfg.n_vspecs = nv;
    cg_plan *p = nullptr;
    cg_status st = cg_plan_create(&cfg, &p);
    if (st != CG_OK)
        return (st == CG_ERR_UNSUPPORTED) ? st : CG_ERR_CORRUPT;
    const uint64_t sb = (uint64_t)get32(h + 40) | ((uint64_t)get32(h + 44) << 32);
    if ((int32_t)get32(h + 36) != p->tp.ngroups || sections(p, sb).end != len) {
        cg_plan_destroy(p);
        return CG_ERR_CORRUPT;
    }
    *plan_out = p;
    if (stream_bytes)
        *stream_bytes = sb;
    return CG_OK;
}

cg_status cg_deserialize(const cg_plan *p, const void *host_in, size_t len,
                         const cg_encoded *dev, cg_stream_t stream)
{
    if (p == nullptr || host_in == nullptr || dev == nullptr)
        return CG_ERR_INVALID_ARG;
    if (!dev->bytestream || !dev->lengths || !dev->cdf || !dev->amax)
        return CG_ERR_INVALID_ARG;
    const uint8_t *h = static_cast<const uint8_t *>(host_in);
    if (len < kHeaderFixed)
        return CG_ERR_CORRUPT;
    const uint64_t sb = (uint64_t)get32(h + 40) | ((uint64_t)get32(h + 44) << 32);
    const Sections sec = sections(p, sb);
    if (sec.end != len)
        return CG_ERR_CORRUPT;
    if (dev->bytestream_capacity < align_up((size_t)sb, 16))
        return CG_ERR_CAPACITY;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dev->amax, h + sec.amax, 4 * (size_t)p->num_streams,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(dev->lengths, h + sec.lengths, 4 * (size_t)p->num_streams,
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(dev->cdf, h + sec.cdf, 2 * (size_t)p->cdf_entries,
                            cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && sb > 0)
        e = cudaMemcpyAsync(dev->bytestream, h + sec.streams, (size_t)sb, cudaMemcpyHostToDevice,
                            s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? CG_OK : CG_ERR_CUDA;
}

cg_status cg_object_range(const cg_plan *p, int32_t object, int32_t *first_token,
                          int32_t *num_tokens)
{
    ObjectRange r;
    if (p == nullptr || !object_range(p, object, &r))
        return CG_ERR_INVALID_ARG;
    if (first_token)
        *first_token = r.t0;
    if (num_tokens)
        *num_tokens = r.n;
    return CG_OK;
}

cg_status cg_object_streams(const cg_plan *p, const void *workspace, int32_t object,
                            uint64_t *offset, uint64_t *bytes, cg_stream_t stream)
{
    ObjectRange r;
    if (p == nullptr || workspace == nullptr || !object_range(p, object, &r))
        return CG_ERR_INVALID_ARG;
    // tile bases are ordered group, K/V, layer and end with the total
    const uint64_t *base = reinterpret_cast<const uint64_t *>(
        static_cast<const uint8_t *>(workspace) + p->ws_tile_base);
    const size_t first = (size_t)r.g0 * 2 * p->L, last = (size_t)(r.g0 + r.ng) * 2 * p->L;
    uint64_t b0 = 0, b1 = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&b0, base + first, 8, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&b1, base + last, 8, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return CG_ERR_CUDA;
    if (b1 < b0)
        return CG_ERR_CORRUPT;
    if (offset)
        *offset = b0;
    if (bytes)
        *bytes = b1 - b0;
    return CG_OK;
}

cg_status cg_object_container_size(const cg_plan *p, int32_t object, uint64_t stream_bytes,
                                   size_t *bytes)
{
    ObjectRange r;
    if (p == nullptr || bytes == nullptr || !object_range(p, object, &r))
        return CG_ERR_INVALID_ARG;
    *bytes = sections_for(p, r.n, r.ng, stream_bytes).end;
    return CG_OK;
}

cg_status cg_serialize_object(const cg_plan *p, const cg_encoded *enc, const void *workspace,
                              int32_t object, void *host_out, size_t host_capacity,
                              size_t *written, cg_stream_t stream)
{
    ObjectRange r;
    if (p == nullptr || enc == nullptr || host_out == nullptr || !object_range(p, object, &r))
        return CG_ERR_INVALID_ARG;
    uint64_t off = 0, sb = 0;
    cg_status st = cg_object_streams(p, workspace, object, &off, &sb, stream);
    if (st != CG_OK)
        return st;
    const Sections sec = sections_for(p, r.n, r.ng, sb);
    if (host_capacity < sec.end)
        return CG_ERR_CAPACITY;
    if (off + sb > enc->bytestream_capacity)
        return CG_ERR_CAPACITY;
    uint8_t *h = static_cast<uint8_t *>(host_out);
    write_header(h, p, r.n, r.ng, sb);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // amax [2][L][T] -> the object's columns, as [2][L][n]
    cudaError_t e = cudaMemcpy2DAsync(h + sec.amax, 4 * (size_t)r.n, enc->amax + r.t0,
                                      4 * (size_t)p->T, 4 * (size_t)r.n, (size_t)2 * p->L,
                                      cudaMemcpyDeviceToHost, s);
    // its streams (and their lengths) and CDF blocks are contiguous
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h + sec.lengths, enc->lengths + (size_t)2 * p->L * r.t0,
                            (size_t)8 * p->L * r.n, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h + sec.cdf, enc->cdf + (size_t)r.g0 * p->tp.cdf_per_group,
                            sec.streams - sec.cdf, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && sb > 0)
        e = cudaMemcpyAsync(h + sec.streams, enc->bytestream + off, (size_t)sb,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return CG_ERR_CUDA;
    if (written)
        *written = sec.end;
    return CG_OK;
}

cg_status cg_deserialize_objects(const cg_plan *p, int32_t n, const void *const *hosts,
                                 const size_t *lens, const cg_encoded *dev,
                                 uint64_t *stream_bytes, cg_stream_t stream)
{
    if (p == nullptr || hosts == nullptr || lens == nullptr || dev == nullptr)
        return CG_ERR_INVALID_ARG;
    if (!dev->bytestream || !dev->lengths || !dev->cdf || !dev->amax)
        return CG_ERR_INVALID_ARG;
    if (n != num_objects(p))
        return CG_ERR_INVALID_ARG;
    // check every header before copying anything
    const size_t hb = header_bytes(p);
    std::vector<uint8_t> want(hb);
    std::vector<uint64_t> sbs(n);
    uint64_t total = 0;
    for (int32_t o = 0; o < n; ++o) {
        ObjectRange r;
        object_range(p, o, &r);
        const uint8_t *h = static_cast<const uint8_t *>(hosts[o]);
        if (h == nullptr)
            return CG_ERR_INVALID_ARG;
        if (lens[o] < hb)
            return CG_ERR_CORRUPT;
        const uint64_t sb = (uint64_t)get32(h + 40) | ((uint64_t)get32(h + 44) << 32);
        write_header(want.data(), p, r.n, r.ng, sb);
        if (memcmp(want.data(), h, hb) != 0 || sections_for(p, r.n, r.ng, sb).end != lens[o])
            return CG_ERR_CORRUPT;
        sbs[o] = sb;
        total += sb;
    }
    if (dev->bytestream_capacity < align_up((size_t)total, 16))
        return CG_ERR_CAPACITY;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    uint64_t off = 0;
    for (int32_t o = 0; o < n && e == cudaSuccess; ++o) {
        ObjectRange r;
        object_range(p, o, &r);
        const uint8_t *h = static_cast<const uint8_t *>(hosts[o]);
        const Sections sec = sections_for(p, r.n, r.ng, sbs[o]);
        e = cudaMemcpy2DAsync(dev->amax + r.t0, 4 * (size_t)p->T, h + sec.amax, 4 * (size_t)r.n,
                              4 * (size_t)r.n, (size_t)2 * p->L, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev->lengths + (size_t)2 * p->L * r.t0, h + sec.lengths,
                                (size_t)8 * p->L * r.n, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev->cdf + (size_t)r.g0 * p->tp.cdf_per_group, h + sec.cdf,
                                sec.streams - sec.cdf, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess && sbs[o] > 0)
            e = cudaMemcpyAsync(dev->bytestream + off, h + sec.streams, (size_t)sbs[o],
                                cudaMemcpyHostToDevice, s);
        off += sbs[o];
    }
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return CG_ERR_CUDA;
    if (stream_bytes)
        *stream_bytes = total;
    return CG_OK;
}

}  // extern "C"

