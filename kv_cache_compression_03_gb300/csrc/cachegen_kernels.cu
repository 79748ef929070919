// CUDA kernels of the CacheGen codec for sm_103a.
//
// Source of the method: "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析"
// (0539edu.com/news/4720135), §2 quantisation, §3 CDF normalisation,
// §4 arithmetic coding in <=256-token batches, §5 prefix-sum decoding and
// dequantisation; the coder is the 32-bit low/high coder with pending bits
// of Witten, Neal & Cleary, CACM 30(6), 1987.
//
// Work decomposition: one CTA of 256 threads per tile = (token group,
// K/V, layer). Encode (one kernel per tile, then a tile scan and a pack):
//   A1  warp per token row: amax over the C channels (16-byte loads, the
//       |x| maximum taken on bf16 bit patterns), scale factor per token;
//   A2  thread per channel pair: quantise every token of the group,
//       histogram in shared memory (each thread owns its channels' rows,
//       so no atomics), write the symbols to a scratch row per stream;
//   B   thread per channel pair: integer CDF in place of the histogram,
//       copied out as the tile's CDF block;
//   C   thread per token: arithmetic-code the token's stream over the C
//       channels with the shared-memory CDF rows, renormalising in bulk
//       (leading-zero counts instead of a bit loop), into a stream slot.
// Pack: block scan of the tile's lengths + the tile's base offset, then
// the slots are copied to their packed position.
// Decode: per tile, the CDF block is staged in shared memory, the lengths
// are scanned, and each thread decodes one stream (binary search of the
// CDF row with the coder's exact multiply-compare), dequantising into the
// bf16 output row.
//
// No kernel waits on another block, and every loop is bounded by the
// tile's token and channel counts.

#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "cg_internal.h"

namespace {

constexpr int NT = CG_TILE_THREADS;
constexpr uint32_t kQuarter = 0x40000000u;

__device__ __forceinline__ void set_status(uint32_t *st, uint32_t code)
{
    atomicCAS(st, 0u, code);
}

struct Tile {
    int32_t g, kv, l, t0, n, N;
    uint64_t first_stream;  // index of the tile's first stream
    uint64_t cdf_base;      // entry offset of the tile's CDF block
};

__device__ __forceinline__ Tile tile_of(const cg_tile_params &P, int32_t tile)
{
    Tile t;
    t.l = tile % P.L;
    t.kv = (tile / P.L) & 1;
    t.g = tile / (2 * P.L);
    // groups: objects of chunk_tokens tokens, each cut into runs of <= 256
    int32_t nf = P.full_objects * P.groups_per_object;
    if (t.g < nf) {
        int32_t o = t.g / P.groups_per_object;
        int32_t j = t.g - o * P.groups_per_object;
        t.t0 = o * P.chunk_tokens + j * CG_GROUP_TOKENS;
        t.n = min(CG_GROUP_TOKENS, P.chunk_tokens - j * CG_GROUP_TOKENS);
    } else {
        int32_t j = t.g - nf;
        int32_t base = P.full_objects * P.chunk_tokens;
        t.t0 = base + j * CG_GROUP_TOKENS;
        t.n = min(CG_GROUP_TOKENS, P.T - base - j * CG_GROUP_TOKENS);
    }
    t.N = P.bins[t.kv][t.l];
    t.first_stream = (uint64_t)2 * P.L * t.t0 + ((uint64_t)t.kv * P.L + t.l) * (uint64_t)t.n;
    t.cdf_base = (uint64_t)t.g * P.cdf_per_group + P.cdf_off[t.kv][t.l];
    return t;
}

// Block-wide exclusive scan of one value per thread (256 threads).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_sums,
                                                         uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = (lane < NT / 32) ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < NT / 32)
            warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    uint32_t before = (warp > 0) ? warp_sums[warp - 1] : 0u;
    if (total)
        *total = warp_sums[NT / 32 - 1];
    return before + x - v;
}

// ------------------------------------------------------------ quantiser

// q = round_half_even(fp32(fp32(x * f) + MAX)), clamped to [0, 2*MAX]
// (the clamp never acts on finite input; it keeps table indices in range
// when the input holds inf/NaN, which is reported separately).
__device__ __forceinline__ uint32_t quantise(float x, float f, float fmax, int32_t two_max)
{
    float y = __fadd_rn(__fmul_rn(x, f), fmax);
    int32_t q = __float2int_rn(y);
    q = max(0, min(q, two_max));
    return (uint32_t)q;
}

// ------------------------------------------------------------ bit writer

struct Enc {
    uint32_t low, high, pending;
    uint32_t nb;        // valid bits in acc (< 32 between calls)
    uint64_t acc;
    uint32_t *out;
    uint32_t nwords, cap_words;
};

// Append m <= 32 bits (v < 2^m), MSB first; whole 32-bit words are stored
// big-endian so that the slot holds the stream's bytes in order.
__device__ __forceinline__ void put_bits(Enc &e, uint64_t v, uint32_t m)
{
    e.acc = (e.acc << m) | v;
    e.nb += m;
    if (e.nb >= 32) {
        e.nb -= 32;
        uint32_t w = (uint32_t)(e.acc >> e.nb);
        if (e.nwords < e.cap_words)
            e.out[e.nwords] = __byte_perm(w, 0, 0x0123);
        e.nwords++;
    }
}

// Rare path: more than 32 bits to emit at once (a long pending run).
__device__ __noinline__ void put_bits_long(Enc &e, uint32_t B, uint32_t n, uint32_t P)
{
    uint32_t b0 = B >> (n - 1);
    put_bits(e, b0, 1);
    while (P > 0) {
        uint32_t c = P < 32u ? P : 32u;
        uint64_t ones = (((uint64_t)1) << c) - 1;
        put_bits(e, b0 ? 0 : ones, c);
        P -= c;
    }
    if (n > 1)
        put_bits(e, B & ((1u << (n - 1)) - 1u), n - 1);
}

// One coder step for the symbol interval [lo, hi) of 2^16 (hi in 1..65536).
// The renormalisation of the textbook coder runs bit by bit: while low and
// high share their top bit, emit it (with the pending bits after the
// first); then, while low = 01.. and high = 10.., drop their second bit and
// count a pending bit. Both runs are counted here with leading-zero counts:
// n shared leading bits, then k underflow positions.
__device__ __forceinline__ void enc_symbol(Enc &e, uint32_t lo, uint32_t hi)
{
    uint32_t d = e.high - e.low;  // range - 1
    uint32_t nlow = e.low + (uint32_t)(((uint64_t)d * lo + lo) >> 16);
    uint32_t nhigh = e.low + (uint32_t)(((uint64_t)d * hi + hi) >> 16) - 1u;
    uint32_t n = __clz(nlow ^ nhigh);
    uint32_t L1 = nlow << n;
    uint32_t H1 = (nhigh << n) | ((1u << n) - 1u);
    uint32_t k = __clz(~((L1 & ~H1) << 1));
    e.low = (L1 << k) & 0x7FFFFFFFu;
    e.high = (H1 << k) | ((1u << k) - 1u) | 0x80000000u;
    uint32_t P = e.pending;
    if (n != 0) {
        uint32_t B = nlow >> (32u - n);
        if (P + n <= 32u) {
            // first bit, P complements of it, then the other n-1 bits: as a
            // number that is B + (2^P - 1) * 2^(n-1)
            uint64_t v = (uint64_t)B + (((((uint64_t)1) << P) - 1) << (n - 1));
            put_bits(e, v, P + n);
        } else {
            put_bits_long(e, B, n, P);
        }
        e.pending = k;
    } else {
        e.pending = P + k;
    }
}

// Termination: one more pending bit, then 0 if low < 1/4 else 1, followed
// by the pending bits; zero-pad and store the last word. Returns the
// stream length in bits.
__device__ __forceinline__ uint32_t enc_finish(Enc &e)
{
    uint32_t P = e.pending + 1;
    uint32_t b = e.low >= kQuarter ? 1u : 0u;
    if (P + 1 <= 32u) {
        put_bits(e, ((((uint64_t)1) << P) - 1) + b, P + 1);
    } else {
        put_bits(e, b, 1);
        while (P > 0) {
            uint32_t c = P < 32u ? P : 32u;
            put_bits(e, b ? 0 : ((((uint64_t)1) << c) - 1), c);
            P -= c;
        }
    }
    uint32_t bits = e.nwords * 32u + e.nb;
    if (e.nb) {
        uint32_t w = (uint32_t)(e.acc << (32u - e.nb));
        if (e.nwords < e.cap_words)
            e.out[e.nwords] = __byte_perm(w, 0, 0x0123);
        e.nwords++;
    }
    return bits;
}

// ---------------------------------------------------------------- encode

__global__ void __launch_bounds__(NT, 3)
    k_encode_tiles(const uint16_t *__restrict__ kv, const cg_tile_params P, uint8_t *sym_ws,
                   float *__restrict__ amax_out, uint16_t *__restrict__ cdf_out,
                   int32_t *__restrict__ lengths, uint8_t *__restrict__ slots,
                   uint32_t *__restrict__ tile_totals, uint32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const Tile tl = tile_of(P, blockIdx.x);
    const int32_t C = P.C;
    const int32_t N = tl.N, Lp = N + 1;
    const int32_t M = N / 2 - 1;
    const float fmax = (float)M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // shared layout: table[C][Lp] u16 (histogram, then CDF), fac[256] f32
    uint16_t *table = reinterpret_cast<uint16_t *>(smem);
    const uint32_t table_bytes = ((uint32_t)C * Lp * 2u + 15u) & ~15u;
    float *fac = reinterpret_cast<float *>(smem + table_bytes);
    __shared__ uint32_t warp_sums[NT / 32];
    __shared__ uint32_t nonfinite;

    if (tid == 0)
        nonfinite = 0;
    {
        uint4 *t4 = reinterpret_cast<uint4 *>(table);
        for (uint32_t i = tid; i < table_bytes / 16; i += NT)
            t4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    const size_t row_stride = (size_t)C;
    const uint16_t *rows = kv + ((size_t)(tl.l * 2 + tl.kv) * P.T + tl.t0) * row_stride;

    // A1: amax per token (warp per row). |x| on bf16 bits is the bit pattern
    // with the sign cleared; finite values order like their patterns.
    for (int t = warp; t < tl.n; t += NT / 32) {
        const uint4 *r4 = reinterpret_cast<const uint4 *>(rows + (size_t)t * row_stride);
        uint32_t m = 0;
        for (int v = lane; v < C / 8; v += 32) {
            uint4 x = __ldg(r4 + v);
            m = __vmaxu2(m, x.x & 0x7FFF7FFFu);
            m = __vmaxu2(m, x.y & 0x7FFF7FFFu);
            m = __vmaxu2(m, x.z & 0x7FFF7FFFu);
            m = __vmaxu2(m, x.w & 0x7FFF7FFFu);
        }
        m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) {
            float a = __uint_as_float(m << 16);
            float f;
            if (m >= 0x7F80u) {  // inf or NaN somewhere in the row
                nonfinite = 1;
                f = 0.0f;
            } else {
                f = (m == 0) ? 0.0f : __fdiv_rn(fmax, a);
            }
            fac[t] = f;
            amax_out[((size_t)tl.kv * P.L + tl.l) * P.T + tl.t0 + t] = a;
        }
    }
    __syncthreads();
    if (tid == 0 && nonfinite)
        set_status(status, CG_ERR_NONFINITE);

    // A2: quantise and count. Thread owns channel pairs p = tid + 256 j;
    // histogram row of channel c is table[c*Lp ...] (Lp odd: the rows of a
    // warp's 32 consecutive pairs start in 32 different banks).
    const int32_t npairs = C / 2;
    uint8_t *sym_tile = sym_ws + tl.first_stream * (uint64_t)C;
    for (int32_t p = tid; p < npairs; p += NT) {
        uint16_t *h0 = table + (size_t)(2 * p) * Lp;
        uint16_t *h1 = h0 + Lp;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(rows) + p;
        uint16_t *dst = reinterpret_cast<uint16_t *>(sym_tile) + p;
        int t = 0;
        for (; t + 4 <= tl.n; t += 4) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                w[u] = __ldg(src + (size_t)(t + u) * (row_stride / 2));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float f = fac[t + u];
                uint32_t q0 = quantise(__uint_as_float(w[u] << 16), f, fmax, 2 * M);
                uint32_t q1 = quantise(__uint_as_float(w[u] & 0xFFFF0000u), f, fmax, 2 * M);
                h0[q0] += 1;
                h1[q1] += 1;
                dst[(size_t)(t + u) * (row_stride / 2)] = (uint16_t)(q0 | (q1 << 8));
            }
        }
        for (; t < tl.n; ++t) {
            uint32_t w = __ldg(src + (size_t)t * (row_stride / 2));
            float f = fac[t];
            uint32_t q0 = quantise(__uint_as_float(w << 16), f, fmax, 2 * M);
            uint32_t q1 = quantise(__uint_as_float(w & 0xFFFF0000u), f, fmax, 2 * M);
            h0[q0] += 1;
            h1[q1] += 1;
            dst[(size_t)t * (row_stride / 2)] = (uint16_t)(q0 | (q1 << 8));
        }
    }

    // B: CDF in place. cdf[i] = floor(cum_i * (65536 - N) / n) + i; the floor
    // uses m = ceil(2^32 / n): cum*K < 2^24 and n <= 256 keep the product's
    // error below 2^-8 <= 1/n, under the quotient's distance to the next
    // integer, so (cum*K*m) >> 32 is the exact floor.
    {
        const uint64_t inv = ((((uint64_t)1) << 32) + (uint64_t)tl.n - 1) / (uint64_t)tl.n;
        const uint32_t K = 65536u - (uint32_t)N;
        for (int32_t p = tid; p < npairs; p += NT) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint16_t *row = table + (size_t)(2 * p + h) * Lp;
                uint32_t cum = 0;
                for (int32_t i = 0; i <= N; ++i) {
                    uint32_t cnt = (i < N) ? row[i] : 0u;
                    uint32_t fl = (uint32_t)(((uint64_t)(cum * K) * inv) >> 32);
                    row[i] = (uint16_t)(fl + (uint32_t)i);  // 65536 wraps to 0
                    cum += cnt;
                }
            }
        }
    }
    __syncthreads();
    {
        // the tile's CDF block: same [C][Lp] layout, 16-byte aligned
        const uint32_t nbytes = (uint32_t)C * Lp * 2u;
        uint4 *dst = reinterpret_cast<uint4 *>(cdf_out + tl.cdf_base);
        const uint4 *src = reinterpret_cast<const uint4 *>(table);
        for (uint32_t i = tid; i < nbytes / 16; i += NT)
            dst[i] = src[i];
    }

    // C: one stream per token
    uint32_t nbytes_stream = 0;
    if (tid < tl.n) {
        Enc e;
        e.low = 0;
        e.high = 0xFFFFFFFFu;
        e.pending = 0;
        e.nb = 0;
        e.acc = 0;
        e.out = reinterpret_cast<uint32_t *>(slots + (tl.first_stream + tid) * (uint64_t)P.slot_stride);
        e.nwords = 0;
        e.cap_words = P.slot_stride / 4;
        const uint8_t *srow = sym_tile + (size_t)tid * C;
        for (int32_t c0 = 0; c0 < C; c0 += 8) {
            uint2 v = *reinterpret_cast<const uint2 *>(srow + c0);
            const uint16_t *trow = table + (size_t)c0 * Lp;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t s = ((j < 4 ? v.x : v.y) >> (8 * (j & 3))) & 0xFFu;
                uint32_t lo = trow[s];
                uint32_t hi = (((uint32_t)trow[s + 1] + 0xFFFFu) & 0xFFFFu) + 1u;  // 0 -> 65536
                enc_symbol(e, lo, hi);
                trow += Lp;
            }
        }
        uint32_t bits = enc_finish(e);
        nbytes_stream = (bits + 7u) / 8u;
        if (e.nwords > e.cap_words)
            set_status(status, CG_ERR_CAPACITY);
        lengths[tl.first_stream + tid] = (int32_t)nbytes_stream;
    }
    uint32_t total = 0;
    block_exclusive_scan(nbytes_stream, warp_sums, &total);
    if (tid == 0)
        tile_totals[blockIdx.x] = total;
}

// Exclusive scan of the per-tile byte totals (one CTA), plus the grand
// total; when expect is given (decode), the total must equal it.
__global__ void __launch_bounds__(1024)
    k_scan_tiles(const uint32_t *__restrict__ totals, int32_t ntiles, uint64_t *__restrict__ base,
                 uint64_t *__restrict__ total_out, int check, uint64_t expect,
                 uint32_t *__restrict__ status)
{
    __shared__ uint64_t wsum[32];
    __shared__ uint64_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        carry_s = 0;
    __syncthreads();
    for (int32_t c0 = 0; c0 < ntiles; c0 += 1024) {
        int32_t i = c0 + tid;
        uint64_t v = (i < ntiles) ? totals[i] : 0;
        uint64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint64_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint64_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o)
                    w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        uint64_t carry = carry_s;
        uint64_t excl = carry + (warp ? wsum[warp - 1] : 0) + x - v;
        if (i < ntiles)
            base[i] = excl;
        __syncthreads();
        if (tid == 0)
            carry_s = carry + wsum[31];
        __syncthreads();
    }
    if (tid == 0) {
        base[ntiles] = carry_s;
        *total_out = carry_s;
        if (check && carry_s != expect)
            set_status(status, CG_ERR_CORRUPT);
    }
}

// Copy each tile's stream slots to their packed position.
__global__ void __launch_bounds__(NT)
    k_pack(const cg_tile_params P, const int32_t *__restrict__ lengths,
           const uint8_t *__restrict__ slots, const uint64_t *__restrict__ tile_base,
           uint8_t *__restrict__ bytestream, uint64_t capacity, uint32_t *__restrict__ status)
{
    __shared__ uint32_t warp_sums[NT / 32];
    __shared__ uint32_t offs[NT];
    const Tile tl = tile_of(P, blockIdx.x);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t len = (tid < tl.n) ? (uint32_t)lengths[tl.first_stream + tid] : 0u;
    uint32_t off = block_exclusive_scan(len, warp_sums, nullptr);
    offs[tid] = off;
    __syncthreads();
    const uint64_t base = tile_base[blockIdx.x];
    for (int i = warp; i < tl.n; i += NT / 32) {
        uint32_t li = (uint32_t)lengths[tl.first_stream + i];
        uint64_t dst = base + offs[i];
        if (li > P.slot_stride || dst + li > capacity) {
            if (lane == 0)
                set_status(status, CG_ERR_CAPACITY);
            continue;
        }
        const uint8_t *src = slots + (tl.first_stream + i) * (uint64_t)P.slot_stride;
        for (uint32_t b = lane; b < li; b += 32)
            bytestream[dst + b] = src[b];
    }
}

// ---------------------------------------------------------------- decode

// Per-tile byte totals of the stream lengths (decode side).
__global__ void __launch_bounds__(NT)
    k_tile_sums(const cg_tile_params P, const int32_t *__restrict__ lengths,
                uint32_t *__restrict__ tile_totals, uint32_t *__restrict__ status)
{
    __shared__ uint32_t warp_sums[NT / 32];
    const Tile tl = tile_of(P, blockIdx.x);
    const int tid = threadIdx.x;
    const int32_t maxlen = 2 * P.C + 2;  // 16 bits per symbol + termination
    uint32_t len = 0;
    if (tid < tl.n) {
        int32_t v = lengths[tl.first_stream + tid];
        if (v < 1 || v > maxlen)
            set_status(status, CG_ERR_CORRUPT);
        else
            len = (uint32_t)v;
    }
    uint32_t total = 0;
    block_exclusive_scan(len, warp_sums, &total);
    if (tid == 0)
        tile_totals[blockIdx.x] = total;
}

struct BitReader {
    const uint8_t *base;
    uint64_t wa;   // next aligned word to load
    uint64_t end;  // stream end (bytes past it read as 0)
    uint64_t buf;  // upcoming bits, MSB first
    int32_t avail;
};

__device__ __forceinline__ uint32_t load_word_be(const uint8_t *base, uint64_t wa, uint64_t end)
{
    if (wa >= end)
        return 0u;
    uint32_t w = __byte_perm(*reinterpret_cast<const uint32_t *>(base + wa), 0, 0x0123);
    uint64_t nv = end - wa;
    if (nv < 4)
        w &= ~(0xFFFFFFFFu >> (8u * (uint32_t)nv));
    return w;
}

__device__ __forceinline__ void br_refill(BitReader &r)
{
    if (r.avail <= 32) {
        r.buf |= (uint64_t)load_word_be(r.base, r.wa, r.end) << (32 - r.avail);
        r.wa += 4;
        r.avail += 32;
    }
}

__device__ __forceinline__ void br_init(BitReader &r, const uint8_t *base, uint64_t sb, uint64_t se)
{
    r.base = base;
    r.end = se;
    r.wa = sb & ~(uint64_t)3;
    uint32_t skip = (uint32_t)(sb - r.wa);
    uint32_t w = load_word_be(base, r.wa, se) << (8u * skip);
    r.buf = (uint64_t)w << 32;
    r.avail = 32 - 8 * (int32_t)skip;
    r.wa += 4;
    br_refill(r);
    br_refill(r);
}

// Take m <= 32 bits.
__device__ __forceinline__ uint32_t br_take(BitReader &r, uint32_t m)
{
    uint32_t v = (uint32_t)((r.buf >> 1) >> (63u - m));
    r.buf <<= m;
    r.avail -= (int32_t)m;
    br_refill(r);
    return v;
}

__global__ void __launch_bounds__(NT, 3)
    k_decode_tiles(const cg_tile_params P, const uint8_t *__restrict__ bytestream,
                   uint64_t stream_bytes, const int32_t *__restrict__ lengths,
                   const uint16_t *__restrict__ cdf, const float *__restrict__ amax,
                   const uint64_t *__restrict__ tile_base, uint16_t *__restrict__ kv_out,
                   uint32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t warp_sums[NT / 32];
    __shared__ float deq[64];
    __shared__ uint32_t bad;
    const Tile tl = tile_of(P, blockIdx.x);
    const int32_t C = P.C;
    const int32_t N = tl.N, Lp = N + 1;
    const int32_t M = N / 2 - 1;
    const int tid = threadIdx.x;
    uint16_t *table = reinterpret_cast<uint16_t *>(smem);

    if (tid == 0)
        bad = 0;
    {
        const uint32_t nb16 = (uint32_t)C * Lp * 2u / 16u;
        const uint4 *src = reinterpret_cast<const uint4 *>(cdf + tl.cdf_base);
        uint4 *dst = reinterpret_cast<uint4 *>(table);
        for (uint32_t i = tid; i < nb16; i += NT)
            dst[i] = __ldg(src + i);
    }
    if (tid < N)
        deq[tid] = __fdiv_rn((float)(tid - M), (float)M);
    uint32_t len = 0;
    if (tid < tl.n) {
        int32_t v = lengths[tl.first_stream + tid];
        len = (v > 0) ? (uint32_t)v : 0u;
    }
    uint32_t off = block_exclusive_scan(len, warp_sums, nullptr);  // has __syncthreads
    // every CDF row must start at 0, end at 65536 (stored 0) and rise strictly
    for (int32_t c = tid; c < C; c += NT) {
        const uint16_t *row = table + (size_t)c * Lp;
        uint32_t ok = (row[0] == 0) && (row[N] == 0);
        for (int32_t i = 1; i < N; ++i)
            ok &= (row[i] > row[i - 1]);
        if (!ok)
            bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0)
            set_status(status, CG_ERR_CORRUPT);
        return;
    }
    if (tid >= tl.n)
        return;

    uint64_t sb = tile_base[blockIdx.x] + off;
    uint64_t se = sb + len;
    if (se > stream_bytes) {
        set_status(status, CG_ERR_CORRUPT);
        se = stream_bytes;
        if (sb > se)
            sb = se;
    }
    BitReader br;
    br_init(br, bytestream, sb, se);
    uint32_t low = 0, high = 0xFFFFFFFFu;
    uint32_t value = br_take(br, 32);
    const float a = amax[((size_t)tl.kv * P.L + tl.l) * P.T + tl.t0 + tid];
    uint16_t *orow = kv_out + ((size_t)(tl.l * 2 + tl.kv) * P.T + tl.t0 + tid) * (size_t)C;
    const uint32_t top_step = 1u << (31 - __clz((uint32_t)(N - 1)));

    for (int32_t c0 = 0; c0 < C; c0 += 8) {
        uint32_t packed[4];
        const uint16_t *row = table + (size_t)c0 * Lp;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t d = high - low;
            uint32_t v = value - low;
            uint32_t s = 0;
            for (uint32_t step = top_step; step != 0; step >>= 1) {
                uint32_t t = s + step;
                if (t < (uint32_t)N) {
                    uint32_t cv = row[t];
                    if ((uint32_t)(((uint64_t)d * cv + cv) >> 16) <= v)
                        s = t;
                }
            }
            uint32_t lo = row[s];
            uint32_t hi = (((uint32_t)row[s + 1] + 0xFFFFu) & 0xFFFFu) + 1u;  // 0 -> 65536
            uint32_t nlow = low + (uint32_t)(((uint64_t)d * lo + lo) >> 16);
            uint32_t nhigh = low + (uint32_t)(((uint64_t)d * hi + hi) >> 16) - 1u;
            uint32_t n = __clz(nlow ^ nhigh);
            uint32_t L1 = nlow << n;
            uint32_t H1 = (nhigh << n) | ((1u << n) - 1u);
            uint32_t k = __clz(~((L1 & ~H1) << 1));
            low = (L1 << k) & 0x7FFFFFFFu;
            high = (H1 << k) | ((1u << k) - 1u) | 0x80000000u;
            uint32_t bits = br_take(br, n + k);
            uint32_t V1 = (value << n) | (bits >> k);
            value = (V1 & 0x80000000u) | ((V1 << k) & 0x7FFFFFFFu) | (bits & ((1u << k) - 1u));
            // dequantise: bf16(fp32((q - MAX) / MAX) * a)
            float y = __fmul_rn(deq[s], a);
            uint32_t yb = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y));
            if (j & 1)
                packed[j >> 1] |= yb << 16;
            else
                packed[j >> 1] = yb;
            row += Lp;
        }
        *reinterpret_cast<uint4 *>(orow + c0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

// The dynamic shared-memory limit is a per-device function attribute: set
// it once per device.
cudaError_t ensure_smem_attributes()
{
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    const uint64_t bit = ((uint64_t)1) << (dev & 63);
    if (done.load() & bit)
        return cudaSuccess;
    err = cudaFuncSetAttribute(k_encode_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               CG_SMEM_LIMIT - 1024);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(k_decode_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   CG_SMEM_LIMIT - 1024);
    if (err == cudaSuccess)
        done.fetch_or(bit);
    return err;
}

}  // namespace

const char *cg_kernel_name(int id)
{
    static const char *names[CG_K_COUNT] = {"k_encode_tiles", "k_scan_tiles(encode)", "k_pack",
                                            "k_tile_sums", "k_scan_tiles(decode)",
                                            "k_decode_tiles"};
    return (id >= 0 && id < CG_K_COUNT) ? names[id] : "unknown";
}

void cg_profiler::begin(int id, cudaStream_t s)
{
    if ((size_t)(used + 1) * 2 > events.size())
        return;
    ids[used] = (int8_t)id;
    cudaEventRecord(events[2 * used], s);
}

void cg_profiler::end(cudaStream_t s)
{
    if ((size_t)(used + 1) * 2 > events.size())
        return;
    cudaEventRecord(events[2 * used + 1], s);
    ++used;
}

int cg_encode_launch_count() { return 3; }
int cg_decode_launch_count() { return 3; }

cudaError_t cg_launch_encode(const cg_plan *p, const void *kv, void *ws, const cg_encoded *out,
                             cudaStream_t stream)
{
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + CG_WS_STATUS);
    uint64_t *total = reinterpret_cast<uint64_t *>(w + CG_WS_TOTAL);
    uint32_t *tile_totals = reinterpret_cast<uint32_t *>(w + p->ws_tile_totals);
    uint64_t *tile_base = reinterpret_cast<uint64_t *>(w + p->ws_tile_base);
    uint8_t *sym = w + p->ws_symbols;
    uint8_t *slots = w + p->ws_slots;
    const int ntiles = p->tp.ntiles;

    cudaError_t err = cudaMemsetAsync(w, 0, CG_WS_STATUS_BYTES, stream);
    if (err != cudaSuccess)
        return err;
    err = ensure_smem_attributes();
    if (err != cudaSuccess)
        return err;
    p->prof.begin(CG_K_ENCODE_TILES, stream);
    k_encode_tiles<<<ntiles, NT, p->smem_encode, stream>>>(
        static_cast<const uint16_t *>(kv), p->tp, sym, out->amax, out->cdf, out->lengths, slots,
        tile_totals, status);
    p->prof.end(stream);
    p->prof.begin(CG_K_SCAN_ENCODE, stream);
    k_scan_tiles<<<1, 1024, 0, stream>>>(tile_totals, ntiles, tile_base, total, 0, 0, status);
    p->prof.end(stream);
    p->prof.begin(CG_K_PACK, stream);
    k_pack<<<ntiles, NT, 0, stream>>>(p->tp, out->lengths, slots, tile_base, out->bytestream,
                                      (uint64_t)out->bytestream_capacity, status);
    p->prof.end(stream);
    return cudaGetLastError();
}

cudaError_t cg_launch_decode(const cg_plan *p, const cg_encoded *in, uint64_t stream_bytes,
                             void *ws, void *kv_out, cudaStream_t stream)
{
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + CG_WS_STATUS);
    uint64_t *total = reinterpret_cast<uint64_t *>(w + CG_WS_TOTAL);
    uint32_t *tile_totals = reinterpret_cast<uint32_t *>(w + p->ws_tile_totals);
    uint64_t *tile_base = reinterpret_cast<uint64_t *>(w + p->ws_tile_base);
    const int ntiles = p->tp.ntiles;

    cudaError_t err = cudaMemsetAsync(w, 0, CG_WS_STATUS_BYTES, stream);
    if (err != cudaSuccess)
        return err;
    err = ensure_smem_attributes();
    if (err != cudaSuccess)
        return err;
    p->prof.begin(CG_K_TILE_SUMS, stream);
    k_tile_sums<<<ntiles, NT, 0, stream>>>(p->tp, in->lengths, tile_totals, status);
    p->prof.end(stream);
    p->prof.begin(CG_K_SCAN_DECODE, stream);
    k_scan_tiles<<<1, 1024, 0, stream>>>(tile_totals, ntiles, tile_base, total, 1, stream_bytes,
                                         status);
    p->prof.end(stream);
    p->prof.begin(CG_K_DECODE_TILES, stream);
    k_decode_tiles<<<ntiles, NT, p->smem_decode, stream>>>(
        p->tp, in->bytestream, stream_bytes, in->lengths, in->cdf, in->amax, tile_base,
        static_cast<uint16_t *>(kv_out), status);
    p->prof.end(stream);
    return cudaGetLastError();
}
