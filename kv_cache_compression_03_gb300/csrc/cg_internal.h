// Internal declarations shared by the codec's host API and its kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "cachegen.h"

// Limits of this build.
#define CG_MAX_LAYERS 256
#define CG_MAX_CHANNELS 4096
// Tokens per group: the encoder works in batches of at most 256 tokens,
// each with its own CDFs ("LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与
// 源码解析", §4).
#define CG_GROUP_TOKENS 256
// Threads per tile CTA: one per token of a group.
#define CG_TILE_THREADS 256
// Shared memory a CTA may use on sm_103a.
#define CG_SMEM_LIMIT (227 * 1024)

// Workspace status block (first 256 bytes of every workspace).
#define CG_WS_STATUS_BYTES 256
#define CG_WS_STATUS 0        // u32 first device error (cg_status), 0 = none
#define CG_WS_TOTAL 8         // u64 total stream bytes

// Per-launch description of the tiles. A tile is one (group, K/V, layer);
// tile index = (group * 2 + kv) * L + layer, which is also the order of
// the tiles' streams, CDF blocks and bytes.
struct cg_tile_params {
    int32_t L, T, C, chunk_tokens;
    int32_t ngroups, ntiles;
    int32_t groups_per_object, full_objects;
    uint64_t cdf_per_group;  // CDF entries of one group (all K/V, layers)
    uint32_t slot_stride;    // bytes of one stream slot in the workspace (16-byte pad first)
    // symbol scratch: the (kv, layer) pairs order[nib_begin, nib_end) (the
    // 16-bin pairs, when C is a multiple of 32 and at least 1024) keep their
    // symbols as 4-bit codes (C/2 bytes per token), all others as bytes; the
    // pairs' regions follow the order of `order`, each T rows long
    int32_t nib_begin, nib_end;
    uint32_t one;  // always 1: a multiplier the decoder's compiler cannot fold
                   // away (its search additions then run on the FMA pipe)
    uint8_t bins[2][CG_MAX_LAYERS];
    uint32_t cdf_off[2][CG_MAX_LAYERS];  // offset of (kv, l) inside a group block
    // (kv, layer) pairs as (kv << 8) | layer, largest bin count first: the
    // tile grid runs through them pair-major, so the heaviest tiles start
    // first and the tail of the launch is light
    uint16_t order[2 * CG_MAX_LAYERS];
};

// Kernel identities for per-kernel timing.
enum cg_kernel_id {
    CG_K_ENCODE_TILES = 0,
    CG_K_SCAN_ENCODE,
    CG_K_PACK,
    CG_K_TILE_SUMS,
    CG_K_SCAN_DECODE,
    CG_K_DECODE_TILES,
    CG_K_COUNT
};

struct cg_profiler {
    std::vector<cudaEvent_t> events;  // 2 per recorded launch
    std::vector<int8_t> ids;
    int32_t used = 0;
    // bracket one launch; both are no-ops when profiling is off or full
    void begin(int id, cudaStream_t s);
    void end(cudaStream_t s);
};

// One launch class: the (kv, layer) pairs order[begin, begin + count) all
// use `bins` bins.
struct cg_bin_class {
    int32_t begin, count, bins;
    size_t smem_encode, smem_decode;
};

// Side stream and fork/join events of a plan, created on first use for
// the device that is current then (recreated if another device is).
struct cg_side_stream {
    int device = -1;
    cudaStream_t stream = nullptr;
    cudaStream_t stream_hi = nullptr;  // the same at the device's greatest priority
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaError_t ensure();
    void release();
};

struct cg_plan {
    int32_t L, T, H, D, C, chunk_tokens;
    std::vector<cg_quant_spec> kspecs, vspecs;
    cg_tile_params tp;
    int32_t max_bins;
    uint64_t num_streams;
    uint64_t cdf_entries;
    // workspace layout (byte offsets)
    size_t ws_tile_totals, ws_tile_base, ws_symbols, ws_slots, ws_bytes;
    size_t max_stream_bytes;
    size_t smem_encode, smem_decode;  // dynamic shared memory (largest class)
    // launch classes, largest bin count first; each class's tiles are one
    // kernel launch sized for that bin count, and the classes run
    // concurrently (a side stream forked from and joined to the caller's)
    std::vector<cg_bin_class> classes;
    mutable cg_side_stream side;
    mutable cg_profiler prof;
};

cudaError_t cg_launch_encode(const cg_plan *p, const void *kv, void *ws, const cg_encoded *out,
                             cudaStream_t stream);
cudaError_t cg_launch_decode(const cg_plan *p, const cg_encoded *in, uint64_t stream_bytes,
                             void *ws, void *kv_out, cudaStream_t stream);
const char *cg_kernel_name(int id);
int cg_encode_launch_count(const cg_plan *p);
int cg_decode_launch_count(const cg_plan *p);
// dynamic shared memory of the tile kernels for C channels and `bins` bins
size_t cg_smem_encode(int32_t C, int32_t bins);
size_t cg_smem_decode(int32_t C, int32_t bins);
// Decoder CDF tables above this many bytes are staged in channel parts so
// that several CTAs fit on an SM; channels per part (C when one part).
#define CG_DECODE_TABLE_BUDGET (36 * 1024)
int32_t cg_decode_part_channels(int32_t C, int32_t bins);
// The encoder's channels per part (rows of at least 1024 channels, a
// multiple of 32; C when one part).
int32_t cg_encode_part_channels(int32_t C, int32_t bins);

// Counting layout of the encoder's phase A for rows of C channels at `bins`
// bins: each counting thread owns W consecutive channels; for rows under
// 4 * CG_TILE_THREADS channels, R groups of C / W threads (R * C / W =
// CG_TILE_THREADS, R <= 8) count different rows into private copies of the
// histogram, which phase B adds up (R copies must fit the table budget).
__host__ __device__ inline void cg_count_layout(int32_t C, int32_t bins, int32_t *W, int32_t *R)
{
    *R = 1;
    if (C >= 4 * CG_TILE_THREADS) {
        *W = 4;
        return;
    }
    const int64_t table = (int64_t)C * (bins + 1) * 2;
    for (int32_t w = 4; w >= 2; w >>= 1) {
        const int32_t u = C / w;
        if (C % w == 0 && u <= CG_TILE_THREADS && CG_TILE_THREADS % u == 0 &&
            CG_TILE_THREADS / u <= 8 && (CG_TILE_THREADS / u) * table <= CG_DECODE_TABLE_BUDGET) {
            *W = w;
            *R = CG_TILE_THREADS / u;
            return;
        }
    }
    *W = (C >= 2 * CG_TILE_THREADS) ? 2 : 1;
}
