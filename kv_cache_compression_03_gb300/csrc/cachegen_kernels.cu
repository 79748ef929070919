// CUDA kernels of the CacheGen codec for sm_103a.
//
// Source of the method: "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析"
// (0539edu.com/news/4720135), §2 quantisation, §3 CDF normalisation,
// §4 arithmetic coding in <=256-token batches, §5 prefix-sum decoding and
// dequantisation; the coder is the 32-bit low/high coder with pending bits
// of Witten, Neal & Cleary, CACM 30(6), 1987.
//
// Work decomposition: one CTA of 256 threads per tile = (token group,
// K/V, layer). Tiles are grouped by bin count; each group is one launch of
// a kernel specialised for 16 or 32 bins (or a generic one) with its own
// shared-memory size and CTAs per SM, and the launches of one call run
// concurrently on the caller's stream and a forked side stream (for the
// encoder, one at the greatest priority, so its 32-bin tiles start first).
// Encode (then a tile scan and a pack):
//   A  16-bin rows counted four channels per thread whose row groups fill
//      the block (1024 channels; 256 in four groups, ...): each thread loads
//      its four channels of eight rows once (the next eight in flight), the
//      row maxima are reduced across the block from those registers, and the
//      same values are quantised (the rounding to an integer as an fp32 addition of
//      1.5 * 2^23), counted into the thread's own shared-memory histogram
//      rows (no atomics) and written to a scratch row per stream as 4-bit
//      codes. Other rows, in blocks of 16: warp per row computes amax over
//      the C channels (16-byte loads; |x| maximum on bf16 bit patterns, one
//      warp reduction) and the row's scale factor; then a thread per four
//      channels re-reads the block (L1/L2-resident), quantises, counts and
//      writes the symbols (4-bit codes for 16 bins, else bytes). The next
//      block's amax overlaps this block's counting. The last read of each
//      raw row carries an L2 evict-first policy, so the streaming rows do
//      not push the scratch out of L2 before phase C reads it back.
//      Rows under 1024 channels are counted by row groups, each group into
//      its own histogram copy (cg_count_layout); at <= 512 channels the
//      maxima of all rows come first and the counting runs without block
//      barriers.
//   B  thread per channel: integer CDF in place of the histogram, copied
//      out as the tile's CDF block.
//   C  thread per token: arithmetic-code the token's stream over the C
//      channels with the shared-memory CDF rows (see Enc); completed words
//      are taken out of the bit buffer once per kStoreEvery symbols.
//   Tables larger than the shared-memory budget (32 and 64 bins at 1024
//   channels) go through phases B and C in channel parts, the coder state
//   carried in registers across a block barrier.
// Pack: block scan of the tile's lengths + the tile's base, then each warp
// copies four streams at a time from their slots to their packed position.
// Decode: per tile, the CDF block (or one channel part at a time) is
// staged in shared memory, the lengths are scanned, and each thread decodes
// one stream (a search of the CDF row against a per-symbol target, checked
// against the coder's exact bounds; the bit buffer refilled once per
// kRefillEvery symbols) and writes the dequantised bf16 row, 16 symbols per
// 32-byte store where the rows allow it (no L1 allocation, L2 evict-first:
// the output is not read again); calls with few tiles split each
// tile's streams over four CTAs. A stream (or part) whose batch of symbols
// over- or under-runs the 64-bit bit buffer (possible only for runs of a
// group's rarest symbols) is redone on an exact path that checks after
// every symbol.
//
// No kernel waits on another block, and every loop is bounded by the
// tile's token and channel counts or the alphabet size.
//
// Test builds only (the product library defines neither): with
// CG_TEST_TARGET_MISS every decoder search target misses, so each symbol
// above the lowest takes the exact re-search; with CG_TEST_EXACT_PATHS the
// encoder codes every stream (and, with channel parts, every part after the
// first) again on its exact path and the decoder decodes every stream (or
// part) again refilling after every symbol. Outputs must not change. With
// CG_TEST_WAIT_TIMEOUT each table copy's barrier expects 16 bytes more than
// the copy brings (the copy itself completes), so the decoder's bounded
// wait runs out and the call reports CG_ERR_TIMEOUT.

#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "cg_internal.h"

namespace {

constexpr int NT = CG_TILE_THREADS;
constexpr int kRowsPerBlock = 16;  // encoder phase A block (two rows per warp)
constexpr int kCountBatch = 8;     // rows whose loads a counting thread keeps in flight

__device__ __forceinline__ void set_status(uint32_t *st, uint32_t code)
{
    atomicCAS(st, 0u, code);
}

// ------------------------------------------------------------ bulk copies
// A tile's CDF rows reach shared memory in one bulk copy (cp.async.bulk:
// the TMA engine, no tensor map) that completes on a shared-memory
// mbarrier, so the CTA's threads do other work meanwhile. Thread 0 issues
// the copy; every thread that reads the table waits on the barrier's phase.

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// thread 0, then a block barrier before the first use
__device__ __forceinline__ void mbar_init(uint64_t *bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Thread 0: copy `bytes` (a multiple of 16) from src (16-byte aligned) to
// dst; completes the barrier's current phase. Earlier reads of dst by the
// block must be ordered before this (a block barrier): the proxy fence then
// orders them before the copy's writes.
__device__ __forceinline__ void bulk_copy_to_smem(void *dst, const void *src, uint32_t bytes,
                                                  uint64_t *bar)
{
#ifdef CG_TEST_WAIT_TIMEOUT
    const uint32_t expect = bytes + 16u;  // a phase that never completes
#else
    const uint32_t expect = bytes;
#endif
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(expect)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Wait until the barrier completes the phase of the given parity; false if
// it has not after kWaitLimit polls (each poll may suspend the thread for a
// while), so a copy that never lands cannot hang the kernel.
#ifdef CG_TEST_WAIT_TIMEOUT
constexpr uint32_t kWaitLimit = 1u << 12;
#else
constexpr uint32_t kWaitLimit = 1u << 20;
#endif
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done)
            return true;
    }
    return false;
}

// Stage a table of `bytes` from src into dst: one bulk copy when src and
// bytes are 16-byte multiples (always, for CDF blocks of a valid plan),
// else a plain copy by all NTH threads (then complete after the caller's
// next block barrier). Returns whether the barrier must be waited on.
template <int NTH>
__device__ __forceinline__ bool stage_table(uint16_t *dst, const uint16_t *src, uint32_t bytes,
                                            uint64_t *bar)
{
    if (((reinterpret_cast<uintptr_t>(src) | bytes) & 15u) == 0) {
        if (threadIdx.x == 0)
            bulk_copy_to_smem(dst, src, bytes, bar);
        return true;
    }
    for (uint32_t i = threadIdx.x; i < bytes / 2; i += NTH)
        dst[i] = src[i];
    return false;
}

struct Tile {
    int32_t index;  // (g * 2 + kv) * L + l
    int32_t g, kv, l, t0, n, N;
    int32_t pair;   // position of (kv, l) in P.order (class launches), else -1
    uint64_t first_stream;  // index of the tile's first stream
    uint64_t cdf_base;      // entry offset of the tile's CDF block
};

__device__ __forceinline__ Tile make_tile(const cg_tile_params &P, int32_t g, int32_t kv,
                                          int32_t l)
{
    Tile t;
    t.g = g;
    t.kv = kv;
    t.l = l;
    t.index = (g * 2 + kv) * P.L + l;
    // groups: objects of chunk_tokens tokens, each cut into runs of <= 256
    const int32_t nf = P.full_objects * P.groups_per_object;
    if (g < nf) {
        const int32_t o = g / P.groups_per_object;
        const int32_t j = g - o * P.groups_per_object;
        t.t0 = o * P.chunk_tokens + j * CG_GROUP_TOKENS;
        t.n = min(CG_GROUP_TOKENS, P.chunk_tokens - j * CG_GROUP_TOKENS);
    } else {
        const int32_t j = g - nf;
        const int32_t base = P.full_objects * P.chunk_tokens;
        t.t0 = base + j * CG_GROUP_TOKENS;
        t.n = min(CG_GROUP_TOKENS, P.T - base - j * CG_GROUP_TOKENS);
    }
    t.N = P.bins[kv][l];
    t.first_stream = (uint64_t)2 * P.L * t.t0 + ((uint64_t)kv * P.L + l) * (uint64_t)t.n;
    t.cdf_base = (uint64_t)g * P.cdf_per_group + P.cdf_off[kv][l];
    t.pair = -1;
    return t;
}

// Tile of block b of a class launch over the pairs order[begin, begin+count)
// (pair-major, group-minor).
__device__ __forceinline__ Tile tile_of_class(const cg_tile_params &P, int32_t begin, int32_t b)
{
    const int32_t i = b / P.ngroups;
    const int32_t g = b - i * P.ngroups;
    const uint32_t kvl = P.order[begin + i];
    Tile t = make_tile(P, g, (int32_t)(kvl >> 8), (int32_t)(kvl & 0xFFu));
    t.pair = begin + i;
    return t;
}

// Tile by its global index (kernels that cover every tile).
__device__ __forceinline__ Tile tile_by_index(const cg_tile_params &P, int32_t index)
{
    return make_tile(P, index / (2 * P.L), (index / P.L) & 1, index % P.L);
}

// Block-wide exclusive scan of one value per thread (NTH threads, a
// multiple of 32 up to 1024).
template <int NTH = NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_sums,
                                                         uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = (lane < NTH / 32) ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < NTH / 32)
            warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const uint32_t before = (warp > 0) ? warp_sums[warp - 1] : 0u;
    if (total)
        *total = warp_sums[NTH / 32 - 1];
    return before + x - v;
}

// The length (clamped at 0) and the byte offset within its tile of the
// stream a decoder thread takes: stream h * NTH + threadIdx.x, the tile's
// streams being split over NT / NTH CTAs of NTH threads. With NTH < NT each
// thread scans NT / NTH consecutive lengths and the offsets go through
// shared memory (offs, NT entries).
template <int NTH>
__device__ __forceinline__ uint32_t tile_stream_offset(const Tile &tl,
                                                       const int32_t *__restrict__ lengths,
                                                       int32_t h, uint32_t *len_out,
                                                       uint32_t *warp_sums, uint32_t *offs)
{
    const int tid = threadIdx.x;
    if (NTH == NT) {
        uint32_t len = 0;
        if (tid < tl.n) {
            const int32_t v = lengths[tl.first_stream + tid];
            len = (v > 0) ? (uint32_t)v : 0u;
        }
        *len_out = len;
        return block_exclusive_scan<NT>(len, warp_sums, nullptr);  // has __syncthreads
    }
    constexpr int K = NT / NTH;
    uint32_t l[K], sum = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int32_t sidx = tid * K + j;
        const int32_t v = (sidx < tl.n) ? lengths[tl.first_stream + sidx] : 0;
        l[j] = (v > 0) ? (uint32_t)v : 0u;
        sum += l[j];
    }
    uint32_t base = block_exclusive_scan<NTH>(sum, warp_sums, nullptr);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        offs[tid * K + j] = base;
        base += l[j];
    }
    __syncthreads();
    const int32_t sidx = h * NTH + tid;
    uint32_t len = 0;
    if (sidx < tl.n) {
        const int32_t v = lengths[tl.first_stream + sidx];
        len = (v > 0) ? (uint32_t)v : 0u;
    }
    *len_out = len;
    return offs[sidx];
}

// ------------------------------------------------------------ quantiser

// q = round_half_even(fp32(fp32(x * f) + MAX)), for finite rows in
// [0, 2*MAX]. The rounding to an integer is one more fp32 addition: y + 1.5 *
// 2^23 lies in [2^23, 2^24), where the spacing of fp32 values is 1, so the
// sum rounds y to the nearest integer with ties to even (1.5 * 2^23 is even)
// and its low mantissa bits hold q (the constant's low 22 bits are zero).
// This keeps the conversion on the FMA pipes instead of the slow
// conversion unit. Returns the sum's bits; the caller masks out q.
__device__ __forceinline__ uint32_t quantise_bits(float x, float f, float fmax)
{
    return __float_as_uint(__fadd_rn(__fadd_rn(__fmul_rn(x, f), fmax), 12582912.0f));
}

// q from quantise_bits. Rows without a usable factor get f = 0 (row_factor)
// and are reported separately; their inf/NaN values give NaN (0 * inf),
// whose bits are not of the form above: the mask keeps q inside the
// alphabet [0, N) for them too (N a power of two: the low log2 N bits;
// otherwise at most N - 1).
template <int NB>
__device__ __forceinline__ uint32_t symbol_of(uint32_t bits, int32_t N)
{
    if (NB > 0 && (NB & (NB - 1)) == 0)
        return bits & (uint32_t)(NB - 1);
    return min(bits & 63u, (uint32_t)(N - 1));
}

// Scale factor MAX / a of a row whose largest |x| has bf16 bits m. A row
// holding inf/NaN, or one so small (a below about 2^-124) that MAX / a
// overflows fp32, has no usable factor: it gets f = 0 and raises the
// non-finite flag, which keeps its symbols in range.
__device__ __forceinline__ float row_factor(uint32_t m, float fmax, uint32_t *nonfinite)
{
    float f = (m == 0) ? 0.0f : __fdiv_rn(fmax, __uint_as_float(m << 16));
    if (m >= 0x7F80u || isinf(f)) {
        *nonfinite = 1;
        f = 0.0f;
    }
    return f;
}

// floor(r * c / 2^16) for r = d + 1 <= 2^32 and c <= 65536, kept mod 2^32
// (it is 2^32 only when r = 2^32 and c = 65536; callers work mod 2^32).
__device__ __forceinline__ uint32_t scale16(uint32_t d, uint32_t c)
{
    return (uint32_t)(((uint64_t)d * c + c) >> 16);
}

// Shifts whose amount may reach 32 (a corrupt stream in the decoder): the
// PTX shifts clamp the amount, so the result is defined (0).
__device__ __forceinline__ uint32_t shl_clamped(uint32_t x, uint32_t s)
{
    uint32_t r;
    asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    return r;
}

__device__ __forceinline__ uint32_t shr_clamped(uint32_t x, uint32_t s)
{
    uint32_t r;
    asm("shr.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    return r;
}

// Renormalisation shift of an interval whose low end (window) is xs and
// whose width - 1 is dn: the number of times the textbook coder doubles the
// interval after this symbol. Renormalisation stops once the width exceeds
// a quarter of the window (2^30) while the interval straddles the middle
// but not the middle half; the width after S doublings is (dn + 1) * 2^S,
// and doubling stops within the first two octaves above 2^30, so S is
// 30 - m or 31 - m with m = msb(dn). After 30 - m doublings the width lies
// in (2^30, 2^31]: the ends xs, hs = xs + dn then sit in quarters whose
// indices differ by 1 or 2, and one more doubling is due exactly when they
// differ by 1 (both ends in one half, or in the middle half), i.e. when bit
// m of xs ^ hs is set. One FLO instead of the two leading-zero counts of
// the textbook bit-by-bit form.
__device__ __forceinline__ uint32_t renorm_shift(uint32_t xs, uint32_t dn)
{
    uint32_t m;
    asm("bfind.u32 %0, %1;" : "=r"(m) : "r"(dn));
    return 30u - m + (shr_clamped(xs ^ (xs + dn), m) & 1u);
}

// ------------------------------------------------------------ encoder

// Coder state in "carry" form. The textbook coder keeps a 32-bit window
// [low, high] and defers the bits of an interval that straddles the middle
// (pending bits). Equivalently, keep the absolute low end of the interval:
// its leading bits are the output, the window x holds its next 32 bits,
// and an addition that overflows x carries into the output bits already
// produced. The renormalisation shift S (the textbook coder's number of
// halvings) is n, the leading bits shared by x and x + range - 1, plus k,
// the following positions where the low end has 1 and the high end 0. The
// textbook window equals x with its top bit cleared (that bit is 1 exactly
// while pending bits are outstanding), so the interval arithmetic and the
// emitted bits are the same as the bit-serial coder's.
struct Enc {
    uint32_t x;       // window of the absolute low end
    uint32_t d;       // range - 1
    uint32_t a0, a1;  // output bits not yet stored: the low nb bits of (a1:a0)
    uint32_t nb;
    uint32_t wp;      // words completed
    uint32_t cap;     // slot capacity in words
    uint32_t hold;    // fast path: the last completed word, not yet stored
    uint32_t flag;    // fast path: a carry ran past the held word
    uint32_t *out;
};

// A carry that ran past every buffered bit goes into the stored words
// (big-endian words). Rare: it needs a run of 1 bits over the whole
// buffer. Takes scalars so that the coder state stays in registers.
__device__ __noinline__ void carry_into_stored(uint32_t *out, uint32_t wp, uint32_t cap,
                                               uint32_t ov)
{
    for (uint32_t i = wp; i > 0 && ov != 0; --i) {
        if (i - 1 >= cap)
            continue;
        const uint32_t w = __byte_perm(out[i - 1], 0, 0x0123);
        const uint32_t s = w + ov;
        ov = (s < w) ? 1u : 0u;
        out[i - 1] = __byte_perm(s, 0, 0x0123);
    }
}

// Take the oldest 32 buffered bits once there are 32. Bits above the
// buffered ones are carries that overflowed the buffer (normally none);
// they belong to the word completed before.
//  - EXACT: store the word now and push such carries into the stored
//    words (a rarely taken branch);
//  - fast path: keep the word in `hold` and store the previously held one,
//    which takes the carries without a branch; a carry through the whole
//    held word only raises `flag`, and the stream is then coded again
//    with the exact path. The fast path has no branch that cannot be
//    predicated, so the unrolled symbol loop stays one block of code.
template <bool EXACT>
__device__ __forceinline__ void enc_store_if_full(Enc &e)
{
    if (e.nb >= 32) {
        e.nb -= 32;
        // nb < 32 here except in a batch that overfilled the buffer (then
        // flagged); the clamping shifts keep that case defined
        const uint32_t ov = __funnelshift_rc(e.a1, 0u, e.nb);  // a1 >> nb
        const uint32_t w = __funnelshift_r(e.a0, e.a1, e.nb);
        if (EXACT) {
            if (ov != 0)
                carry_into_stored(e.out, e.wp, e.cap, ov);
            if (e.wp < e.cap)
                e.out[e.wp] = __byte_perm(w, 0, 0x0123);
        } else {
            // out[-1] lies in the slot's pad: the store needs no test for
            // the first word, only a clamp against the capacity
            const uint32_t prev = e.hold + ov;
            e.flag |= (prev < ov) ? 1u : 0u;
            e.out[(int32_t)min(e.wp, e.cap) - 1] = __byte_perm(prev, 0, 0x0123);
            e.hold = w;
        }
        e.wp++;
        e.a1 = 0;
        e.a0 &= ~__funnelshift_lc(0u, 0xFFFFFFFFu, e.nb);  // the low nb bits
    }
}

// x + t with the carry added into the buffered output (a1:a0).
__device__ __forceinline__ uint32_t add_with_carry(uint32_t x, uint32_t t, uint32_t &a0,
                                                   uint32_t &a1)
{
    uint32_t xs;
    asm("add.cc.u32 %0, %3, %4;\n\t"
        "addc.cc.u32 %1, %1, 0;\n\t"
        "addc.u32 %2, %2, 0;"
        : "=r"(xs), "+r"(a0), "+r"(a1)
        : "r"(x), "r"(t));
    return xs;
}

// Symbols per store check in the fast path. A symbol the encoder codes
// occurs in its group, so its frequency is >= 256 of 2^16 and it adds at most
// 9 bits (1.6 on average here). Fewer than 32 bits are left after a check, so
// a batch overfills the 64-bit buffer (60 bits plus room for the batch's
// carries above them) only if its symbols are nearly all among their groups'
// rarest. The check flags that case and the stream is coded again on the
// exact path, which checks after every symbol.
constexpr int kStoreEvery = 4;

// One symbol with CDF bounds c0 < c1 (c1 in 1..65535: the encoder never
// codes the top symbol, whose upper bound would be 65536). STORE: take a
// completed word out of the buffer afterwards.
template <bool EXACT, bool STORE = true>
__device__ __forceinline__ void enc_symbol(Enc &e, uint32_t c0, uint32_t c1)
{
    const uint32_t t0 = scale16(e.d, c0);
    const uint32_t t1 = scale16(e.d, c1);
    const uint32_t xs = add_with_carry(e.x, t0, e.a0, e.a1);
    const uint32_t dn = t1 - t0 - 1u;  // new range - 1
    const uint32_t S = renorm_shift(xs, dn);
    e.a1 = __funnelshift_l(e.a0, e.a1, S);
    e.a0 = __funnelshift_l(xs, e.a0, S);
    e.x = shl_clamped(xs, S);
    e.d = __funnelshift_l(0xFFFFFFFFu, dn, S);
    e.nb += S;
    if (STORE) {
        if (!EXACT && kStoreEvery > 1)
            e.flag |= (e.nb > 60u) ? 1u : 0u;
        enc_store_if_full<EXACT>(e);
    }
}

// Termination: the code value is the frame start plus 1/4 of the window
// (when the textbook window's low end is below 1/4) or plus 1/2, i.e. two
// more bits, (x >> 30) + 1 with its carry. Stores what is left (the last
// word zero-padded) and returns the stream length in bits.
template <bool EXACT>
__device__ __forceinline__ uint32_t enc_finish(Enc &e)
{
    const uint32_t w2 = (e.x >> 30) + 1u;
    const uint32_t cy = w2 >> 2;
    const uint32_t a0c = e.a0 + cy;
    e.a1 += (a0c < cy) ? 1u : 0u;
    e.a1 = __funnelshift_l(a0c, e.a1, 2);
    e.a0 = (a0c << 2) | (w2 & 3u);
    e.nb += 2;
    enc_store_if_full<EXACT>(e);
    const uint32_t bits = e.wp * 32u + e.nb;
    const uint32_t ov = __funnelshift_r(e.a0, e.a1, e.nb);  // nb < 32
    if (EXACT) {
        if (ov != 0)
            carry_into_stored(e.out, e.wp, e.cap, ov);
    } else {
        const uint32_t prev = e.hold + ov;
        e.flag |= (prev < ov) ? 1u : 0u;
        e.out[(int32_t)min(e.wp, e.cap) - 1] = __byte_perm(prev, 0, 0x0123);
    }
    if (e.nb) {
        const uint32_t w = __funnelshift_lc(0u, e.a0, 32u - e.nb);  // a0 << (32 - nb)
        if (e.wp < e.cap)
            e.out[e.wp] = __byte_perm(w, 0, 0x0123);
        e.wp++;
    }
    return bits;
}

__device__ __forceinline__ void enc_init(Enc &e, uint32_t *out, uint32_t cap)
{
    e.x = 0;
    e.d = 0xFFFFFFFFu;
    e.a0 = e.a1 = 0;
    e.nb = 0;
    e.wp = 0;
    e.cap = cap;
    e.hold = 0;
    e.flag = 0;
    e.out = out;
}

// Code symbols [c_begin, c_begin + C) of a token's symbol row with the CDF
// rows table[0..C) (row j for symbol c_begin + j). c_begin is a multiple of
// 32. Reads 16 symbols per load (bytes, C a multiple of 16) or 32 (4-bit
// codes, C a multiple of 32), else 8.
template <bool EXACT, bool NIB>
__device__ __forceinline__ void code_symbols(Enc &e, const uint8_t *srow8, int32_t c_begin,
                                             int32_t C, const uint16_t *table, int32_t Lp)
{
    const uint16_t *trow = table;
    if (NIB) {
        // 4-bit codes, 32 per 16-byte load (C is a multiple of 32): byte k
        // of a word holds channels 2k (low half) and 2k + 1 (high half)
        const uint4 *srow = reinterpret_cast<const uint4 *>(srow8 + c_begin / 2);
        uint4 next = srow[0];
        for (int32_t c0 = 0; c0 < C; c0 += 32) {
            const uint4 v = next;
            if (c0 + 32 < C)
                next = srow[(c0 >> 5) + 1];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const uint32_t word = (j < 8) ? v.x : (j < 16) ? v.y : (j < 24) ? v.z : v.w;
                const uint32_t half = (j & 1) ? ((word >> 4) & 0x0F0F0F0Fu) : (word & 0x0F0F0F0Fu);
                const uint32_t s = __byte_perm(half, 0, 0x4440 + ((j >> 1) & 3));
                if (EXACT || (j % kStoreEvery) == kStoreEvery - 1)
                    enc_symbol<EXACT, true>(e, trow[s], trow[s + 1]);
                else
                    enc_symbol<EXACT, false>(e, trow[s], trow[s + 1]);
                trow += Lp;
            }
        }
    } else if ((C & 15) == 0) {
        const uint4 *srow = reinterpret_cast<const uint4 *>(srow8 + c_begin);
        uint4 next = srow[0];
        for (int32_t c0 = 0; c0 < C; c0 += 16) {
            const uint4 v = next;
            if (c0 + 16 < C)
                next = srow[(c0 >> 4) + 1];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t word = (j < 4) ? v.x : (j < 8) ? v.y : (j < 12) ? v.z : v.w;
                const uint32_t s = __byte_perm(word, 0, 0x4440 + (j & 3));
                // s <= 2*MAX = N - 2, so cdf[s + 1] is never the top entry
                // (65536, stored as 0)
                if (EXACT || (j % kStoreEvery) == kStoreEvery - 1)
                    enc_symbol<EXACT, true>(e, trow[s], trow[s + 1]);
                else
                    enc_symbol<EXACT, false>(e, trow[s], trow[s + 1]);
                trow += Lp;
            }
        }
    } else {
        const uint2 *srow = reinterpret_cast<const uint2 *>(srow8 + c_begin);
        uint2 next = srow[0];
        for (int32_t c0 = 0; c0 < C; c0 += 8) {
            const uint2 v = next;
            if (c0 + 8 < C)
                next = srow[(c0 >> 3) + 1];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t s = __byte_perm(j < 4 ? v.x : v.y, 0, 0x4440 + (j & 3));
                if (EXACT || (j % kStoreEvery) == kStoreEvery - 1)
                    enc_symbol<EXACT, true>(e, trow[s], trow[s + 1]);
                else
                    enc_symbol<EXACT, false>(e, trow[s], trow[s + 1]);
                trow += Lp;
            }
        }
    }
}

// Code one token's stream: symbols srow[0..C) with the CDF rows of the
// shared table. Returns the length in bits; *flag is set when the fast
// path met a carry it cannot place (then the caller codes it again with
// EXACT).
template <bool EXACT, bool NIB>
__device__ __forceinline__ uint32_t code_stream(const uint8_t *srow8, int32_t C,
                                                const uint16_t *table, int32_t Lp, uint32_t *out,
                                                uint32_t cap, uint32_t *wp_out, uint32_t *flag)
{
    Enc e;
    enc_init(e, out, cap);
    code_symbols<EXACT, NIB>(e, srow8, 0, C, table, Lp);
    const uint32_t bits = enc_finish<EXACT>(e);
    *wp_out = e.wp;
    *flag = e.flag;
    return bits;
}

// The exact path, kept out of line: it runs only for streams where the
// fast path raised its flag. Returns (words << 32) | bits.
template <bool NIB>
__device__ __noinline__ uint64_t code_stream_exact(const uint8_t *srow8, int32_t C,
                                                   const uint16_t *table, int32_t Lp,
                                                   uint32_t *out, uint32_t cap)
{
    uint32_t flag = 0, wp = 0;
    const uint32_t bits = code_stream<true, NIB>(srow8, C, table, Lp, out, cap, &wp, &flag);
    return ((uint64_t)wp << 32) | bits;
}

// Parts path: the fast state `st` raised its flag while coding a part (or
// while finishing); code that part again exactly from the state `st` held at
// the part's start. In the fast state the last completed word is held in a
// register, not stored: store it, then continue in the exact form (which
// stores every word and pushes carries into stored words).
template <bool NIB>
__device__ __noinline__ void code_part_exact(Enc *st, const uint8_t *srow8, int32_t c_begin,
                                             int32_t C, const uint16_t *table, int32_t Lp,
                                             bool from_fast)
{
    Enc e = *st;
    if (from_fast && e.wp >= 1 && e.wp - 1 < e.cap)
        e.out[e.wp - 1] = __byte_perm(e.hold, 0, 0x0123);
    code_symbols<true, NIB>(e, srow8, c_begin, C, table, Lp);
    *st = e;
}

__device__ __noinline__ uint32_t finish_exact(Enc *st)
{
    Enc e = *st;
    const uint32_t bits = enc_finish<true>(e);
    *st = e;
    return bits;
}

// Loads of raw rows read for the last time (the counting passes). They
// carry an L2 evict-first policy: 1.75 GB of rows stream through L2 in a
// 16K-token call, and with the default policy they push out the symbol
// scratch that the same tiles read back in phase C.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint2 ldg_last(const uint2 *a, uint64_t pol)
{
    uint2 r;
    asm("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
        : "=r"(r.x), "=r"(r.y)
        : "l"(a), "l"(pol));
    return r;
}

__device__ __forceinline__ uint32_t ldg_last(const uint32_t *a, uint64_t pol)
{
    uint32_t r;
    asm("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(a), "l"(pol));
    return r;
}

// Phase A, counting one block of rows: each thread owns W consecutive
// channels (W = 4 with 8-byte loads and 4-byte symbol stores; W = 2 and 1
// for narrower rows).
template <int NB, int W, bool NIB, bool PARTIAL = false>
__device__ __forceinline__ void count_block(const uint16_t *__restrict__ rows, int32_t C,
                                            int32_t r0, int32_t nr, const float *fac, float fmax,
                                            uint16_t *table, int32_t N, uint8_t *sym_tile,
                                            int32_t cnt_units = 0)
{
    const int32_t Lp = N + 1;
    const int32_t units = C / W;
    for (int32_t p = threadIdx.x; p < units; p += NT) {
        // PARTIAL: only units below cnt_units count (the table holds their
        // rows); every unit stores its symbols
        uint16_t *h0 = table + (size_t)(W * (PARTIAL ? min(p, cnt_units - 1) : p)) * Lp;
        const bool cnt = !PARTIAL || p < cnt_units;
        for (int32_t rb = r0; rb < r0 + nr; rb += kCountBatch) {
            const int32_t nb = min(kCountBatch, r0 + nr - rb);
            if (W == 4 && nb == kCountBatch) {
                // a full batch: no per-row predicates, addresses from one base
                const uint2 *src = reinterpret_cast<const uint2 *>(rows) + p + (size_t)rb * (C / 4);
                const uint64_t pol = policy_evict_first();
                uint2 w[kCountBatch];
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u)
                    w[u] = ldg_last(src + (size_t)u * (C / 4), pol);
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u) {
                    const float f = fac[rb + u];
                    const uint32_t b0 = quantise_bits(__uint_as_float(w[u].x << 16), f, fmax);
                    const uint32_t b1 = quantise_bits(__uint_as_float(w[u].x & 0xFFFF0000u), f, fmax);
                    const uint32_t b2 = quantise_bits(__uint_as_float(w[u].y << 16), f, fmax);
                    const uint32_t b3 = quantise_bits(__uint_as_float(w[u].y & 0xFFFF0000u), f, fmax);
                    const uint32_t q0 = symbol_of<NB>(b0, N), q1 = symbol_of<NB>(b1, N);
                    const uint32_t q2 = symbol_of<NB>(b2, N), q3 = symbol_of<NB>(b3, N);
                    if (cnt) {
                        h0[q0] += 1;
                        h0[Lp + q1] += 1;
                        h0[2 * Lp + q2] += 1;
                        h0[3 * Lp + q3] += 1;
                    }
                    if (NIB) {
                        // four 4-bit codes, channel 4p + i in bits 4i..4i+3
                        // (multiply-adds: q < 16 leaves no carry between codes)
                        reinterpret_cast<uint16_t *>(sym_tile)[p + (size_t)(rb + u) * (C / 4)] =
                            (uint16_t)(q0 + 16u * q1 + 256u * q2 + 4096u * q3);
                    } else {
                        reinterpret_cast<uint32_t *>(sym_tile)[p + (size_t)(rb + u) * (C / 4)] =
                            __byte_perm(__byte_perm(q0, q1, 0x0040), __byte_perm(q2, q3, 0x0040), 0x5410);
                    }
                }
            } else if (W == 4) {
                const uint2 *src = reinterpret_cast<const uint2 *>(rows) + p;
                uint32_t *dst = reinterpret_cast<uint32_t *>(sym_tile) + p;
                uint2 w[kCountBatch];
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u)
                    w[u] = (u < nb) ? __ldg(src + (size_t)(rb + u) * (C / 4)) : make_uint2(0u, 0u);
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u) {
                    if (u < nb) {
                        const float f = fac[rb + u];
                        const uint32_t q0 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x << 16), f, fmax), N);
                        const uint32_t q1 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x & 0xFFFF0000u), f, fmax), N);
                        const uint32_t q2 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y << 16), f, fmax), N);
                        const uint32_t q3 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y & 0xFFFF0000u), f, fmax), N);
                        if (cnt) {
                            h0[q0] += 1;
                            h0[Lp + q1] += 1;
                            h0[2 * Lp + q2] += 1;
                            h0[3 * Lp + q3] += 1;
                        }
                        if (NIB)
                            reinterpret_cast<uint16_t *>(sym_tile)[p + (size_t)(rb + u) * (C / 4)] =
                                (uint16_t)(q0 | (q1 << 4) | (q2 << 8) | (q3 << 12));
                        else
                            dst[(size_t)(rb + u) * (C / 4)] =
                                __byte_perm(__byte_perm(q0, q1, 0x0040), __byte_perm(q2, q3, 0x0040), 0x5410);
                    }
                }
            } else if (W == 2) {
                const uint32_t *src = reinterpret_cast<const uint32_t *>(rows) + p;
                uint16_t *dst = reinterpret_cast<uint16_t *>(sym_tile) + p;
                uint32_t w[kCountBatch];
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u)
                    w[u] = (u < nb) ? __ldg(src + (size_t)(rb + u) * (C / 2)) : 0u;
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u) {
                    if (u < nb) {
                        const float f = fac[rb + u];
                        const uint32_t q0 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u] << 16), f, fmax), N);
                        const uint32_t q1 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u] & 0xFFFF0000u), f, fmax), N);
                        if (cnt) {
                            h0[q0] += 1;
                            h0[Lp + q1] += 1;
                        }
                        dst[(size_t)(rb + u) * (C / 2)] = (uint16_t)(q0 | (q1 << 8));
                    }
                }
            } else {
                const uint16_t *src = rows + p;
                uint8_t *dst = sym_tile + p;
                uint32_t w[kCountBatch];
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u)
                    w[u] = (u < nb) ? (uint32_t)__ldg(src + (size_t)(rb + u) * C) : 0u;
#pragma unroll
                for (int u = 0; u < kCountBatch; ++u) {
                    if (u < nb) {
                        const uint32_t q = symbol_of<NB>(quantise_bits(__uint_as_float(w[u] << 16), fac[rb + u], fmax), N);
                        if (cnt)
                            h0[q] += 1;
                        dst[(size_t)(rb + u) * C] = (uint8_t)q;
                    }
                }
            }
        }
    }
}

// Phase A, counting one block of rows for rows under 4 * NT channels
// (cg_count_layout): R groups of U = C / W threads; group g counts rows
// r0 + g, r0 + g + R, ... of the block into its own copy of the histogram
// (copy g at table + g * C * Lp) and stores their symbols.
template <int NB, int W, bool NIB, int R>
__device__ __forceinline__ void count_block_groups(const uint16_t *__restrict__ rows, int32_t C,
                                                   int32_t r0, int32_t nr, const float *fac,
                                                   float fmax, uint16_t *table, int32_t N,
                                                   uint8_t *sym_tile)
{
    const int32_t Lp = N + 1;
    const int32_t U = C / W;
    const int32_t g = threadIdx.x / U, p = threadIdx.x - g * U;
    uint16_t *h0 = table + (size_t)g * C * Lp + (size_t)(W * p) * Lp;
    constexpr int kRows = kRowsPerBlock / R;
    const uint64_t pol = policy_evict_first();
    if (W == 4) {
        const uint2 *src = reinterpret_cast<const uint2 *>(rows) + p;
        uint2 w[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int32_t r = r0 + g + R * u;
            w[u] = (r < r0 + nr) ? ldg_last(src + (size_t)r * (C / 4), pol) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int32_t r = r0 + g + R * u;
            if (r < r0 + nr) {
                const float f = fac[r];
                const uint32_t q0 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x << 16), f, fmax), N);
                const uint32_t q1 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x & 0xFFFF0000u), f, fmax), N);
                const uint32_t q2 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y << 16), f, fmax), N);
                const uint32_t q3 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y & 0xFFFF0000u), f, fmax), N);
                h0[q0] += 1;
                h0[Lp + q1] += 1;
                h0[2 * Lp + q2] += 1;
                h0[3 * Lp + q3] += 1;
                if (NIB)
                    reinterpret_cast<uint16_t *>(sym_tile)[p + (size_t)r * (C / 4)] =
                        (uint16_t)(q0 + 16u * q1 + 256u * q2 + 4096u * q3);
                else
                    reinterpret_cast<uint32_t *>(sym_tile)[p + (size_t)r * (C / 4)] =
                        __byte_perm(__byte_perm(q0, q1, 0x0040), __byte_perm(q2, q3, 0x0040), 0x5410);
            }
        }
    } else {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(rows) + p;
        uint32_t w[kRows];
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int32_t r = r0 + g + R * u;
            w[u] = (r < r0 + nr) ? ldg_last(src + (size_t)r * (C / 2), pol) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kRows; ++u) {
            const int32_t r = r0 + g + R * u;
            if (r < r0 + nr) {
                const float f = fac[r];
                const uint32_t q0 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u] << 16), f, fmax), N);
                const uint32_t q1 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u] & 0xFFFF0000u), f, fmax), N);
                h0[q0] += 1;
                h0[Lp + q1] += 1;
                reinterpret_cast<uint16_t *>(sym_tile)[p + (size_t)r * (C / 2)] = (uint16_t)(q0 | (q1 << 8));
            }
        }
    }
}

// Phase A, largest |x| of one row (one warp) as bf16 bits, in every lane:
// the lanes' maxima over the bf16 bit patterns with the sign cleared
// (finite values order like their patterns), then one warp reduction.
__device__ __forceinline__ uint32_t absmax_reduce(uint32_t m)
{
    return __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
}

__device__ __forceinline__ uint32_t row_absmax(const uint16_t *__restrict__ row, int32_t C)
{
    const int lane = threadIdx.x & 31;
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
    uint32_t m = 0;
    for (int v = lane; v < C / 8; v += 32) {
        const uint4 x = __ldg(r4 + v);
        m = __vmaxu2(m, x.x & 0x7FFF7FFFu);
        m = __vmaxu2(m, x.y & 0x7FFF7FFFu);
        m = __vmaxu2(m, x.z & 0x7FFF7FFFu);
        m = __vmaxu2(m, x.w & 0x7FFF7FFFu);
    }
    return absmax_reduce(m);
}

// Phase A, amax of one row in two halves: amax_issue starts the row's
// loads (rows of at most 1024 channels: 4 x 16 bytes per lane) so that they
// are in flight while the block before is counted; amax_finish reduces them.
__device__ __forceinline__ void amax_issue(const uint16_t *__restrict__ row, int32_t C,
                                           bool valid, uint4 (&x)[4])
{
    const int lane = threadIdx.x & 31;
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = lane + 32 * i;
        x[i] = (valid && v < C / 8) ? __ldg(r4 + v) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ uint32_t amax_finish(const uint4 (&x)[4])
{
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = __vmaxu2(m, x[i].x & 0x7FFF7FFFu);
        m = __vmaxu2(m, x[i].y & 0x7FFF7FFFu);
        m = __vmaxu2(m, x[i].z & 0x7FFF7FFFu);
        m = __vmaxu2(m, x[i].w & 0x7FFF7FFFu);
    }
    return absmax_reduce(m);
}

// The scale and factor of two rows a warp has reduced (rows ra and rb with
// maxima ma and mb, in every lane): lane 0 takes ra and lane 1 rb, so the
// two divisions run as one instruction sequence.
__device__ __forceinline__ void store_factors(int32_t ra, uint32_t ma, int32_t rb, uint32_t mb,
                                              int32_t n, float fmax, float *fac, float *amax_row,
                                              uint32_t *nonfinite)
{
    const int lane = threadIdx.x & 31;
    const int32_t r = lane ? rb : ra;
    const uint32_t m = lane ? mb : ma;
    if (lane < 2 && r < n) {
        fac[r] = row_factor(m, fmax, nonfinite);
        amax_row[r] = __uint_as_float(m << 16);
    }
}

// Phase A for 16-bin tiles counted four channels per thread with 4-bit
// symbols, when R row groups of C/4 threads fill the block (C * R = 4 * NT:
// 1024 channels with R = 1, 256 with R = 4, ...): the tile's raw data is
// read once. Thread (g, p) of row group g holds channels 4p..4p+3 of rows
// r0 + uR + g, u < 8, of each batch of 8R rows in registers (the next
// batch's loads already in flight); the row maxima are reduced across the
// block from those registers (a warp reduction, then the warp maxima of the
// row's group), and the same registers are then quantised and counted into
// the group's histogram copy. Two block barriers per batch.
template <int NB, int R>
__device__ __forceinline__ void count_tile_single_read(const uint16_t *__restrict__ rows,
                                                       int32_t C, int32_t n, float fmax,
                                                       float *fac, float *amax_row,
                                                       uint32_t *nonfinite, uint16_t *table,
                                                       int32_t N, uint8_t *sym_tile)
{
    constexpr int U = NT / R;      // threads per row group
    constexpr int WPG = U / 32;    // warps per row group
    static_assert(U % 32 == 0, "a row group is whole warps");
    __shared__ uint32_t wmax[NT / 32][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = tid / U, p = tid % U;
    const int32_t Lp = N + 1;
    uint16_t *h0 = table + (size_t)g * C * Lp + (size_t)(4 * p) * Lp;
    const uint2 *src = reinterpret_cast<const uint2 *>(rows) + p;
    const uint64_t pol = policy_evict_first();
    uint2 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int32_t row = u * R + g;
        w[u] = (row < n) ? ldg_last(src + (size_t)row * (C / 4), pol) : make_uint2(0u, 0u);
    }
    for (int32_t r0 = 0; r0 < n; r0 += 8 * R) {
        uint2 wn[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t row = r0 + 8 * R + u * R + g;
            wn[u] = (row < n) ? ldg_last(src + (size_t)row * (C / 4), pol) : make_uint2(0u, 0u);
        }
        // |x| maxima on bf16 bit patterns: per thread, per warp, per row
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t m = __vmaxu2(w[u].x & 0x7FFF7FFFu, w[u].y & 0x7FFF7FFFu);
            const uint32_t mw = absmax_reduce(m);
            if (lane == 0)
                wmax[warp][u] = mw;
        }
        __syncthreads();
        if (tid < 8 * R) {  // one thread per row of the batch
            const int u = tid / R, gg = tid % R;
            const int32_t row = r0 + u * R + gg;
            if (row < n) {
                uint32_t m = 0;
#pragma unroll
                for (int i = 0; i < WPG; ++i)
                    m = max(m, wmax[gg * WPG + i][u]);
                fac[row] = row_factor(m, fmax, nonfinite);
                amax_row[row] = __uint_as_float(m << 16);
            }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int32_t row = r0 + u * R + g;
            if (row < n) {
                const float f = fac[row];
                const uint32_t q0 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x << 16), f, fmax), N);
                const uint32_t q1 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].x & 0xFFFF0000u), f, fmax), N);
                const uint32_t q2 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y << 16), f, fmax), N);
                const uint32_t q3 = symbol_of<NB>(quantise_bits(__uint_as_float(w[u].y & 0xFFFF0000u), f, fmax), N);
                h0[q0] += 1;
                h0[Lp + q1] += 1;
                h0[2 * Lp + q2] += 1;
                h0[3 * Lp + q3] += 1;
                reinterpret_cast<uint16_t *>(sym_tile)[p + (size_t)row * (C / 4)] =
                    (uint16_t)(q0 + 16u * q1 + 256u * q2 + 4096u * q3);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            w[u] = wn[u];
    }
    __syncthreads();  // every count is in before phase B reads the table
}

// Ask L2 for rows [r, r + nr) of the tile (one contiguous range).
__device__ __forceinline__ void prefetch_rows(const uint16_t *rows, int32_t C, int32_t r,
                                              int32_t nr)
{
    if (nr <= 0)
        return;
    const char *base = reinterpret_cast<const char *>(rows + (size_t)r * C);
    const uint32_t lines = ((uint32_t)nr * (uint32_t)C * 2u + 127u) / 128u;
    for (uint32_t i = threadIdx.x; i < lines; i += NT)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 128u * i));
}

// Phase B for rows [0, nrows) of the table: the integer CDF in place of the
// histogram. cdf[i] = floor(cum_i * (65536 - N) / n) + i; the floor uses
// m = ceil(2^32 / n): cum*K < 2^24 and n <= 256 keep the product's error
// below 2^-8 <= 1/n, under the quotient's distance to the next integer, so
// (cum*K*m) >> 32 is the exact floor.
// With R > 1 the counts are the sum of R histogram copies, nrows * Lp
// entries apart (the CDF goes to copy 0).
__device__ __forceinline__ void cdf_rows(uint16_t *table, int32_t nrows, int32_t N, int32_t n,
                                         int32_t R = 1)
{
    const int32_t Lp = N + 1;
    const uint64_t inv = ((((uint64_t)1) << 32) + (uint64_t)n - 1) / (uint64_t)n;
    const uint32_t K = 65536u - (uint32_t)N;
    const size_t copy = (size_t)nrows * Lp;
    for (int32_t c = threadIdx.x; c < nrows; c += NT) {
        uint16_t *row = table + (size_t)c * Lp;
        uint32_t cum = 0;
#pragma unroll
        for (int32_t i = 0; i <= N; ++i) {
            uint32_t cnt = 0;
            if (i < N) {
                cnt = row[i];
                for (int32_t g = 1; g < R; ++g)
                    cnt += row[i + g * copy];
            }
            const uint32_t fl = (uint32_t)(((uint64_t)(cum * K) * inv) >> 32);
            row[i] = (uint16_t)(fl + (uint32_t)i);  // 65536 wraps to 0
            cum += cnt;
        }
    }
}

// Copy rows [0, nrows) of the table (16-byte multiple) to dst.
__device__ __forceinline__ void copy_rows_out(uint16_t *dst, const uint16_t *table, int32_t nrows,
                                              int32_t Lp)
{
    const uint32_t nbytes = (uint32_t)nrows * Lp * 2u;
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    const uint4 *s4 = reinterpret_cast<const uint4 *>(table);
    for (uint32_t i = threadIdx.x; i < nbytes / 16; i += NT)
        d4[i] = s4[i];
}

// Inf/NaN values of a reported row quantise to the top symbol N - 1
// (symbol_of); its upper bound cdf[N] = 65536 is held as 0 in the table.
// Coding such a tile (its output is undefined) with 65535 as that bound
// keeps every interval well formed: the top symbol then occurs, so
// cdf[N - 1] <= 65534 and its width stays >= 1 of 2^16.
__device__ __forceinline__ void patch_top_bounds(uint16_t *table, int32_t nrows, int32_t N)
{
    __syncthreads();
    for (int32_t c = threadIdx.x; c < nrows; c += NT)
        table[(size_t)c * (N + 1) + N] = 0xFFFFu;
    __syncthreads();
}

// One tile of the encoder. NB > 0 fixes the bin count at compile time
// (16 and 32 are the presets); NB = 0 reads it from the tile. PARTS (rows
// of at least 1024 channels whose CDF table exceeds the shared-memory
// budget): the table holds part_ch channels at a time (a multiple of 32).
// Phase A stores every symbol but counts only the first part; each later
// part is counted from the stored symbols. Each part's CDF rows are built,
// copied out and used to code that part's channels of every stream, the
// coder state staying in registers across a block barrier; a stream whose
// fast path raised its flag in a part codes that part again exactly from
// the state it held at the part's start, and the rest exactly.
template <int NB, bool PARTS, bool GROUPS>
__device__ __forceinline__ void encode_tile(const Tile &tl, const uint16_t *__restrict__ kv,
                                            const cg_tile_params &P, uint8_t *sym_ws,
                                            float *__restrict__ amax_out,
                                            uint16_t *__restrict__ cdf_out,
                                            int32_t *__restrict__ lengths,
                                            uint8_t *__restrict__ slots,
                                            uint32_t *__restrict__ tile_totals,
                                            uint32_t *__restrict__ status, uint8_t *smem,
                                            uint32_t *warp_sums, uint32_t *nonfinite,
                                            int32_t part_ch)
{
    const int32_t C = P.C;
    const int32_t N = NB > 0 ? NB : tl.N;
    const int32_t Lp = N + 1;
    const float fmax = (float)(N / 2 - 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t tab_ch = PARTS ? part_ch : C;
    int32_t cw = 4, cr = 1;  // counting layout (cg_count_layout; GROUPS: cr > 1)
    if (!PARTS)
        cg_count_layout(C, N, &cw, &cr);
    if (!GROUPS)
        cr = 1;

    // shared: cr x table[tab_ch][Lp] u16 (histogram copies; then the CDF in
    // copy 0) | fac[256] f32
    uint16_t *table = reinterpret_cast<uint16_t *>(smem);
    const uint32_t table_bytes = ((uint32_t)cr * tab_ch * Lp * 2u + 15u) & ~15u;
    float *fac = reinterpret_cast<float *>(smem + table_bytes);

    if (tid == 0)
        *nonfinite = 0;
    {
        uint4 *t4 = reinterpret_cast<uint4 *>(table);
        for (uint32_t i = tid; i < table_bytes / 16; i += NT)
            t4[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const uint16_t *rows = kv + ((size_t)(tl.l * 2 + tl.kv) * P.T + tl.t0) * (size_t)C;
    float *amax_row = amax_out + ((size_t)tl.kv * P.L + tl.l) * P.T + tl.t0;
    // symbol rows: the pair's region (T rows, pairs in the order of
    // P.order, 4-bit codes for pairs in [nib_begin, nib_end)), then the
    // group's rows from its first token
    const bool nib = NB == 16 && tl.pair >= P.nib_begin && tl.pair < P.nib_end;
    const uint32_t row_bytes = nib ? (uint32_t)C / 2 : (uint32_t)C;
    const int32_t nib_before = min(max(tl.pair - P.nib_begin, 0), P.nib_end - P.nib_begin);
    uint8_t *sym_tile = sym_ws + (uint64_t)P.T * ((uint64_t)C * tl.pair - (uint64_t)(C / 2) * nib_before) +
                        (uint64_t)tl.t0 * row_bytes;
    const int32_t nblocks = (tl.n + kRowsPerBlock - 1) / kRowsPerBlock;

    if (NB == 16 && !PARTS && nib && cw == 4 && C * cr == 4 * NT) {
        // 4-bit symbols, four channels per thread, the row groups fill the block
        if (cr == 1)
            count_tile_single_read<NB, 1>(rows, C, tl.n, fmax, fac, amax_row, nonfinite, table,
                                          N, sym_tile);
        else if (GROUPS && cr == 2)
            count_tile_single_read<NB, 2>(rows, C, tl.n, fmax, fac, amax_row, nonfinite, table,
                                          N, sym_tile);
        else if (GROUPS && cr == 4)
            count_tile_single_read<NB, 4>(rows, C, tl.n, fmax, fac, amax_row, nonfinite, table,
                                          N, sym_tile);
        else if (GROUPS && cr == 8)
            count_tile_single_read<NB, 8>(rows, C, tl.n, fmax, fac, amax_row, nonfinite, table,
                                          N, sym_tile);
    } else if (GROUPS && C <= 512) {
        // A for rows of at most 512 channels counted by row groups (a tile of
        // at most 256 KB, which stays in L2 between the passes): the maxima
        // and factors of all rows first (a warp per two rows at a time), then
        // every row counted, with no block barriers in between (each thread
        // owns its histogram rows)
        for (int32_t ra = 2 * warp; ra < tl.n; ra += NT / 16) {
            const int32_t rb = ra + 1;
            const uint32_t ma = row_absmax(rows + (size_t)ra * C, C);
            const uint32_t mb = (rb < tl.n) ? row_absmax(rows + (size_t)rb * C, C) : 0u;
            store_factors(ra, ma, rb, mb, tl.n, fmax, fac, amax_row, nonfinite);
        }
        __syncthreads();
        for (int32_t b = 0; b < nblocks; ++b) {
            const int32_t r0 = b * kRowsPerBlock;
            const int32_t nr = min(kRowsPerBlock, tl.n - r0);
            if (cw == 4) {
                if (cr == 2) {
                    if (nib)
                        count_block_groups<NB, 4, true, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                    else
                        count_block_groups<NB, 4, false, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                } else if (cr == 4) {
                    if (nib)
                        count_block_groups<NB, 4, true, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                    else
                        count_block_groups<NB, 4, false, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                } else {
                    if (nib)
                        count_block_groups<NB, 4, true, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                    else
                        count_block_groups<NB, 4, false, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                }
            } else {
                if (cr == 2)
                    count_block_groups<NB, 2, false, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                else if (cr == 4)
                    count_block_groups<NB, 2, false, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                else
                    count_block_groups<NB, 2, false, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            }
        }
        __syncthreads();
    } else {
    // A: amax of block 0; then per step, count block b while the loads for
    // block b + 1's amax are in flight (one row per warp), and ask L2 for
    // block b + 2
    {
        // rows warp and warp + 8 of block 0
        const int32_t ra = warp, rb = warp + NT / 32;
        const uint32_t ma = (ra < tl.n) ? row_absmax(rows + (size_t)ra * C, C) : 0u;
        const uint32_t mb = (rb < tl.n) ? row_absmax(rows + (size_t)rb * C, C) : 0u;
        store_factors(ra, ma, rb, mb, tl.n, fmax, fac, amax_row, nonfinite);
    }
    __syncthreads();
    const bool pipelined = (C <= 1024);
    for (int32_t b = 0; b < nblocks; ++b) {
        const int32_t r0 = b * kRowsPerBlock;
        const int32_t nr = min(kRowsPerBlock, tl.n - r0);
        const int32_t r2 = r0 + 2 * kRowsPerBlock;
        prefetch_rows(rows, C, r2, min(kRowsPerBlock, tl.n - r2));
        const int32_t ta = r0 + kRowsPerBlock + warp;
        uint4 xa[4];
        if (pipelined)
            amax_issue(rows + (size_t)ta * C, C, ta < tl.n, xa);
        if (PARTS) {
            if (nib)
                count_block<NB, 4, true, true>(rows, C, r0, nr, fac, fmax, table, N, sym_tile,
                                               part_ch / 4);
            else
                count_block<NB, 4, false, true>(rows, C, r0, nr, fac, fmax, table, N, sym_tile,
                                                part_ch / 4);
        } else if (!GROUPS || cr == 1) {
            if (nib)
                count_block<NB, 4, true>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            else if (cw == 4)
                count_block<NB, 4, false>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            else if (cw == 2)
                count_block<NB, 2, false>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            else
                count_block<NB, 1, false>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
        } else if (cw == 4) {
            if (cr == 2) {
                if (nib)
                    count_block_groups<NB, 4, true, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                else
                    count_block_groups<NB, 4, false, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            } else if (cr == 4) {
                if (nib)
                    count_block_groups<NB, 4, true, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                else
                    count_block_groups<NB, 4, false, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            } else {
                if (nib)
                    count_block_groups<NB, 4, true, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
                else
                    count_block_groups<NB, 4, false, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            }
        } else {
            if (cr == 2)
                count_block_groups<NB, 2, false, 2>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            else if (cr == 4)
                count_block_groups<NB, 2, false, 4>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
            else
                count_block_groups<NB, 2, false, 8>(rows, C, r0, nr, fac, fmax, table, N, sym_tile);
        }
        const uint32_t ma = pipelined ? amax_finish(xa)
                                      : (ta < tl.n) ? row_absmax(rows + (size_t)ta * C, C) : 0u;
        const int32_t tb = ta + NT / 32;
        const uint32_t mb = (tb < tl.n) ? row_absmax(rows + (size_t)tb * C, C) : 0u;
        store_factors(ta, ma, tb, mb, tl.n, fmax, fac, amax_row, nonfinite);
        __syncthreads();
    }
    }
    if (tid == 0 && *nonfinite)
        set_status(status, CG_ERR_NONFINITE);

    uint32_t nbytes_stream = 0;
    const uint32_t cap = (P.slot_stride - 16) / 4;
    uint32_t *out = reinterpret_cast<uint32_t *>(slots + (tl.first_stream + tid) * (uint64_t)P.slot_stride + 16);
    const uint8_t *srow = sym_tile + (size_t)tid * row_bytes;
    if (!PARTS) {
        // B: CDF in place, copied out as the tile's CDF block ([C][Lp],
        // 16-byte aligned)
        cdf_rows(table, C, N, tl.n, cr);
        __syncthreads();
        copy_rows_out(cdf_out + tl.cdf_base, table, C, Lp);
        if (*nonfinite)
            patch_top_bounds(table, C, N);

        // C: one stream per token
        if (tid < tl.n) {
            uint32_t wp = 0, flag = 0;
            uint32_t bits = nib ? code_stream<false, true>(srow, C, table, Lp, out, cap, &wp, &flag)
                                : code_stream<false, false>(srow, C, table, Lp, out, cap, &wp, &flag);
#ifdef CG_TEST_EXACT_PATHS
            flag = 1;
#endif
            if (flag) {
                const uint64_t r = nib ? code_stream_exact<true>(srow, C, table, Lp, out, cap)
                                       : code_stream_exact<false>(srow, C, table, Lp, out, cap);
                bits = (uint32_t)r;
                wp = (uint32_t)(r >> 32);
            }
            nbytes_stream = (bits + 7u) / 8u;
            if (wp > cap)
                set_status(status, CG_ERR_CAPACITY);
            lengths[tl.first_stream + tid] = (int32_t)nbytes_stream;
        }
    } else {
        const bool active = tid < tl.n;
        Enc e;
        enc_init(e, out, cap);
        bool exact = false;
        uint32_t bits = 0;
        for (int32_t c_begin = 0; c_begin < C; c_begin += part_ch) {
            const int32_t nch = min(part_ch, C - c_begin);
            if (c_begin > 0) {
                // count this part from the stored symbols
                __syncthreads();  // the previous part's coding is done with the table
                {
                    uint4 *t4 = reinterpret_cast<uint4 *>(table);
                    for (uint32_t i = tid; i < table_bytes / 16; i += NT)
                        t4[i] = make_uint4(0, 0, 0, 0);
                }
                __syncthreads();
                for (int32_t u = c_begin / 4 + tid; u < (c_begin + nch) / 4; u += NT) {
                    uint16_t *h0 = table + (size_t)(4 * u - c_begin) * Lp;
                    for (int32_t r = 0; r < tl.n; ++r) {
                        const uint8_t *rp = sym_tile + (size_t)r * row_bytes;
                        uint32_t q0, q1, q2, q3;
                        if (nib) {
                            const uint32_t w = reinterpret_cast<const uint16_t *>(rp)[u];
                            q0 = w & 15u;
                            q1 = (w >> 4) & 15u;
                            q2 = (w >> 8) & 15u;
                            q3 = w >> 12;
                        } else {
                            const uint32_t w = reinterpret_cast<const uint32_t *>(rp)[u];
                            q0 = w & 0xFFu;
                            q1 = (w >> 8) & 0xFFu;
                            q2 = (w >> 16) & 0xFFu;
                            q3 = w >> 24;
                        }
                        h0[q0] += 1;
                        h0[Lp + q1] += 1;
                        h0[2 * Lp + q2] += 1;
                        h0[3 * Lp + q3] += 1;
                    }
                }
                __syncthreads();
            }
            cdf_rows(table, nch, N, tl.n);
            __syncthreads();
            copy_rows_out(cdf_out + tl.cdf_base + (size_t)c_begin * Lp, table, nch, Lp);
            if (*nonfinite)
                patch_top_bounds(table, nch, N);
            if (active) {
                const bool last = c_begin + nch >= C;
                if (!exact) {
                    const Enc save = e;
                    if (nib)
                        code_symbols<false, true>(e, srow, c_begin, nch, table, Lp);
                    else
                        code_symbols<false, false>(e, srow, c_begin, nch, table, Lp);
                    if (last)
                        bits = enc_finish<false>(e);
#ifdef CG_TEST_EXACT_PATHS
                    if (c_begin > 0)
                        e.flag = 1;
#endif
                    if (e.flag) {
                        e = save;
                        exact = true;
                        if (nib)
                            code_part_exact<true>(&e, srow, c_begin, nch, table, Lp, true);
                        else
                            code_part_exact<false>(&e, srow, c_begin, nch, table, Lp, true);
                        if (last)
                            bits = finish_exact(&e);
                    }
                } else {
                    if (nib)
                        code_part_exact<true>(&e, srow, c_begin, nch, table, Lp, false);
                    else
                        code_part_exact<false>(&e, srow, c_begin, nch, table, Lp, false);
                    if (last)
                        bits = finish_exact(&e);
                }
            }
        }
        if (active) {
            nbytes_stream = (bits + 7u) / 8u;
            if (e.wp > cap)
                set_status(status, CG_ERR_CAPACITY);
            lengths[tl.first_stream + tid] = (int32_t)nbytes_stream;
        }
    }
    uint32_t total = 0;
    block_exclusive_scan(nbytes_stream, warp_sums, &total);
    if (tid == 0)
        tile_totals[tl.index] = total;
}

// Encoder tiles of one launch class (NB bins; 0 = any), at least MINB
// CTAs per SM; PARTS as in encode_tile; GROUPS: rows counted by row groups
// (cg_count_layout gives R > 1).
template <int NB, int MINB, bool PARTS, bool GROUPS>
__global__ void __launch_bounds__(NT, MINB)
    k_encode_class(const uint16_t *__restrict__ kv, const cg_tile_params P, int32_t cls_begin,
                   uint8_t *sym_ws, float *__restrict__ amax_out, uint16_t *__restrict__ cdf_out,
                   int32_t *__restrict__ lengths, uint8_t *__restrict__ slots,
                   uint32_t *__restrict__ tile_totals, uint32_t *__restrict__ status,
                   int32_t part_ch)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t warp_sums[NT / 32];
    __shared__ uint32_t nonfinite;
    const Tile tl = tile_of_class(P, cls_begin, blockIdx.x);
    encode_tile<NB, PARTS, GROUPS>(tl, kv, P, sym_ws, amax_out, cdf_out, lengths, slots,
                                   tile_totals, status, smem, warp_sums, &nonfinite, part_ch);
}

// Exclusive scan of the per-tile byte totals (one CTA), plus the grand
// total; when check is set (decode), the total must equal expect.
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
        const int32_t i = c0 + tid;
        const uint64_t v = (i < ntiles) ? totals[i] : 0;
        uint64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
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
                const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o)
                    w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const uint64_t carry = carry_s;
        const uint64_t excl = carry + (warp ? wsum[warp - 1] : 0) + x - v;
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

// Copy each tile's stream slots to their packed position. A warp moves four
// streams at a time, eight lanes each, so that the load latencies of four
// streams overlap (streams are short: 40-200 bytes in the workloads here).
__global__ void __launch_bounds__(NT)
    k_pack(const cg_tile_params P, const int32_t *__restrict__ lengths,
           const uint8_t *__restrict__ slots, const uint64_t *__restrict__ tile_base,
           uint8_t *__restrict__ bytestream, uint64_t capacity, uint32_t *__restrict__ status)
{
    __shared__ uint32_t warp_sums[NT / 32];
    __shared__ uint32_t offs[NT];
    const Tile tl = tile_by_index(P, blockIdx.x);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t len = (tid < tl.n) ? (uint32_t)lengths[tl.first_stream + tid] : 0u;
    offs[tid] = block_exclusive_scan(len, warp_sums, nullptr);
    __syncthreads();
    const uint64_t base = tile_base[blockIdx.x];
    constexpr int kGroup = 4;          // streams per warp step
    const int sub = lane >> 3;         // this lane's stream within the step
    const uint32_t sl = lane & 7;      // lane within the stream's eight
    for (int32_t i0 = warp * kGroup; i0 < tl.n; i0 += (NT / 32) * kGroup) {
        const int32_t i = i0 + sub;
        uint32_t li = 0;
        uint64_t dst = base;
        if (i < tl.n) {
            li = (uint32_t)lengths[tl.first_stream + i];
            dst = base + offs[i];
            if (li > P.slot_stride - 16 || dst + li > capacity) {
                if (sl == 0)
                    set_status(status, CG_ERR_CAPACITY);
                li = 0;
            }
        }
        const uint8_t *src = slots + (tl.first_stream + (i < tl.n ? i : 0)) * (uint64_t)P.slot_stride + 16;
        // bytes up to the first 4-byte boundary of the destination and after
        // its last one go byte by byte (those words may hold a neighbouring
        // stream's bytes); the body goes as whole words, each taken from two
        // aligned source words by a funnel shift (the slot is 16-byte aligned
        // and holds a multiple of 4 bytes, so no read leaves it)
        const uint32_t h = min((4u - (uint32_t)(dst & 3u)) & 3u, li);
        const uint32_t nw = (li - h) >> 2;
        const uint32_t t0 = h + 4u * nw;
        if (sl < h)
            bytestream[dst + sl] = src[sl];
        if (sl < li - t0)
            bytestream[dst + t0 + sl] = src[t0 + sl];
        uint32_t *d32 = reinterpret_cast<uint32_t *>(bytestream + dst + h);
        const uint32_t *s32 = reinterpret_cast<const uint32_t *>(src);
        // up to four words per lane loaded before any is stored
        for (uint32_t j0 = 0; j0 < nw; j0 += 32) {
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t j = j0 + sl + 8u * k;
                lo[k] = (j < nw) ? s32[j] : 0u;
                hi[k] = (j < nw && h) ? s32[j + 1] : 0u;  // bytes h + 4j .. h + 4j + 3
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t j = j0 + sl + 8u * k;
                if (j < nw)
                    d32[j] = __funnelshift_r(lo[k], hi[k], 8u * h);
            }
        }
    }
}

// ---------------------------------------------------------------- decode

// Per-tile byte totals of the stream lengths (decode side).
__global__ void __launch_bounds__(NT)
    k_tile_sums(const cg_tile_params P, const int32_t *__restrict__ lengths,
                uint32_t *__restrict__ tile_totals, uint32_t *__restrict__ status)
{
    __shared__ uint32_t warp_sums[NT / 32];
    const Tile tl = tile_by_index(P, blockIdx.x);
    const int tid = threadIdx.x;
    const int32_t maxlen = 2 * P.C + 2;  // 16 bits per symbol + termination
    uint32_t len = 0;
    if (tid < tl.n) {
        const int32_t v = lengths[tl.first_stream + tid];
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

// Bit reader over one stream: the next `avail` bits are the top bits of
// (b1:b0) and the bits below them are zero. Offsets are 32-bit, relative
// to the aligned word where the stream starts. Past the stream's end the
// reader goes on into whatever follows (the next stream, or the buffer's
// last word again at its end): a terminated stream decodes to the same
// symbols whatever bits follow it, so those bits need no masking; loads
// are only clamped to stay inside the buffer.
struct Bits {
    const uint8_t *base;  // aligned start of the stream's first word
    uint32_t pos;         // next word to load (bytes from base)
    uint32_t lim;         // last loadable word (bytes from base)
    uint32_t b1, b0;
    int32_t avail;
};

__device__ __forceinline__ uint32_t bits_word(const Bits &r)
{
    return __byte_perm(*reinterpret_cast<const uint32_t *>(r.base + min(r.pos, r.lim)), 0, 0x0123);
}

__device__ __forceinline__ void bits_refill(Bits &r)
{
    if (r.avail <= 32) {  // every valid bit is in b1 and b0 is zero
        const uint32_t w = bits_word(r);
        r.b1 |= __funnelshift_rc(w, 0u, (uint32_t)r.avail);  // w >> avail, 0 when avail = 32
        r.b0 = w << (32 - r.avail);
        r.pos += 4;
        r.avail += 32;
    }
}

// sb: the stream's first byte; words may be loaded up to `last` (the
// buffer's last whole word).
__device__ __forceinline__ void bits_init(Bits &r, const uint8_t *bytestream, uint64_t sb,
                                          uint64_t last)
{
    const uint64_t wa = sb & ~(uint64_t)3;
    r.base = bytestream + wa;
    r.pos = 0;
    r.lim = (uint32_t)(last - wa);
    const uint32_t skip = (uint32_t)(sb - wa);
    r.b1 = bits_word(r) << (8u * skip);
    r.b0 = 0;
    r.avail = 32 - 8 * (int32_t)skip;
    r.pos = 4;
    bits_refill(r);
}

// Drop S bits (S <= 18 for a valid stream, <= 32 for a corrupt one).
__device__ __forceinline__ void bits_skip(Bits &r, uint32_t S)
{
    r.b1 = __funnelshift_l(r.b0, r.b1, S);
    r.b0 = shl_clamped(r.b0, S);
    r.avail -= (int32_t)S;
    bits_refill(r);
}

// Refill for the batched loop below: avail may have gone negative there (a
// batch needed more bits than were buffered; that stream is decoded again),
// so both shifts clamp. nw holds the word at r.pos as loaded (byte order not
// yet swapped); the load of the following one is issued here, a refill
// ahead of its use.
__device__ __forceinline__ void bits_refill_next(Bits &r, uint32_t &nw)
{
    if (r.avail <= 32) {
        const uint32_t w = __byte_perm(nw, 0, 0x0123);
        r.b1 |= __funnelshift_rc(w, 0u, (uint32_t)r.avail);        // w >> avail
        r.b0 = __funnelshift_lc(0u, w, (uint32_t)(32 - r.avail));  // w << (32 - avail)
        r.pos += 4;
        r.avail += 32;
        nw = *reinterpret_cast<const uint32_t *>(r.base + min(r.pos, r.lim));
    }
}

// Symbols per bit-buffer refill in the decoder's main loop. After a refill
// the buffer holds at least 32 bits. A symbol that occurs in its group has
// frequency >= (65536 - N) / 256 of 2^16, so it takes at most 10 bits, and
// four of them fit unless all four are among the group's rarest; a batch that
// does run short is detected (the count of buffered bits goes negative) and
// the stream is decoded again refilling after every symbol.
constexpr int kRefillEvery = 4;

// Search target. The decoder wants the largest s with floor(r * cdf[s] /
// 2^16) <= v (r = d + 1, the coder's own comparison). As cdf[s] < 2^16 that
// holds exactly when cdf[s] <= T = floor(((v + 1) 2^16 - 1) / r), so one
// target per symbol replaces a 64-bit product per probe. The estimate below
// is round(v 2^16 / r) from d and v converted to floats (rounded toward
// zero) and an approximate reciprocal of d; for a valid stream (r > 2^30)
// it is T or T + 1. The caller checks the symbol found against the exact
// bounds and searches again with the exact comparison when they disagree, so
// any error in the estimate costs time, never a wrong symbol.
__device__ __forceinline__ uint32_t search_target(uint32_t d, uint32_t v)
{
    float rc;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(__uint2float_rz(d)));
    // v / d < 4 even for a corrupt stream, so y stays in [128, 256), where
    // the float spacing is 2^-16: adding 1.5 * 2^7 rounds v / d to a multiple
    // of 2^-16, and the low mantissa bits of y are then round(v 2^16 / d)
    const float y = __fmaf_rn(__uint2float_rz(v), rc, 192.0f);
#ifdef CG_TEST_TARGET_MISS
    return 0u * __float_as_uint(y);
#endif
    return __float_as_uint(y) - 0x43400000u;  // the bits of 192.0f
}

// Shared-memory loads at 32-bit shared addresses (volatile: the decoder
// stages a new table between calls in the channel-part kernels).
__device__ __forceinline__ uint32_t lds_u16(uint32_t a)
{
    uint32_t r;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}

__device__ __forceinline__ float lds_f32(uint32_t a)
{
    float r;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(a));
    return r;
}

// sb += inc when e <= T (sb: a search position, here the shared address of
// the current entry). `one` is 1 but comes from the kernel's arguments,
// so the predicated add compiles to a multiply-add on the FMA pipe and stays
// off the integer ALU pipe, the decoder's busiest.
__device__ __forceinline__ void probe_add(uint32_t &sb, uint32_t e, uint32_t T, uint32_t one,
                                          uint32_t inc)
{
    asm("{\n\t.reg .pred p;\n\tsetp.le.u32 p, %1, %2;\n\t@p mad.lo.u32 %0, %3, %4, %0;\n\t}"
        : "+r"(sb)
        : "r"(e), "r"(T), "r"(one), "r"(inc));
}

// One level of the search at entries q, 2q and 3q above the current one
// (p: its shared address; entries are 2 bytes). The three loads are
// independent; as the row rises, the number of entries <= T is the quarter
// to take. Tracking the address itself leaves every probe a load at p plus a
// constant.
__device__ __forceinline__ void search_4way(uint32_t &p, uint32_t q, uint32_t T, uint32_t one)
{
    const uint32_t e1 = lds_u16(p + 2 * q);
    const uint32_t e2 = lds_u16(p + 4 * q);
    const uint32_t e3 = lds_u16(p + 6 * q);
    probe_add(p, e1, T, one, 2 * q);
    probe_add(p, e2, T, one, 2 * q);
    probe_add(p, e3, T, one, 2 * q);
}

__device__ __forceinline__ void search_2way(uint32_t &p, uint32_t q, uint32_t T, uint32_t one)
{
    probe_add(p, lds_u16(p + 2 * q), T, one, 2 * q);
}

// Decode one stream (C symbols with the CDF rows of `table`) and write its
// dequantised row. R > 1 refills the bit buffer once per R symbols and
// returns 1 when a batch ran short of bits (the output is then wrong and the
// caller decodes the stream again with R = 1, which never runs short: a
// symbol takes at most 18 bits and the buffer holds at least 33 after every
// refill).
// Decoder state: x = window of the absolute low end, d = range - 1,
// v = code value - low end, and the bit reader.
struct DecState {
    uint32_t x, d, v;
    Bits br;
};

__device__ __forceinline__ void dec_start(DecState &st, const Bits &br)
{
    st.x = 0;
    st.d = 0xFFFFFFFFu;
    st.v = br.b1;
    st.br = br;
    bits_skip(st.br, 16);
    bits_skip(st.br, 16);
}

// The largest s in [0, N - 1) with floor(r * cdf[s] / 2^16) <= v by the
// coder's own comparison (the byte offset 2s; NB = 0: any N, top_step the
// largest power of two below N).
template <int NB>
__device__ __forceinline__ uint32_t exact_search(const char *rb, uint32_t d, uint32_t v, int32_t N,
                                                 uint32_t top_step)
{
    uint32_t sb = 0;
#pragma unroll 1
    for (uint32_t step = NB > 0 ? (uint32_t)NB / 2 : top_step; step != 0; step >>= 1) {
        const uint32_t t = sb + 2 * step;
        if ((NB > 0 || t < 2 * (uint32_t)N) &&
            scale16(d, *reinterpret_cast<const uint16_t *>(rb + t)) <= v)
            sb = t;
    }
    return sb;
}

// Decode the next C symbols of a stream with the CDF rows of `table` (row c
// for the c-th of them) and write their dequantised values to orow[0, C).
// The search compares against a target (search_target): 16 bins in one
// 4-way level (its loads depend on nothing but the row, so they issue
// early) and two binary ones, or with WIDE two 4-way levels (fewer
// dependent shared-memory round trips, for calls with too few streams to
// hide latency); 32 bins in two 4-way levels and a binary one; other counts
// (NB = 0) in binary steps. `one` must be 1 (see probe_add); `table` and
// `deq` are in shared memory.
// Output: KB symbols per store, 16 (one 32-byte store, a whole DRAM sector;
// C a multiple of 16 and orow 32-byte aligned) or 8 (16 bytes). A sector
// written in two halves some symbols apart is merged in L2, which fills
// from DRAM the halves it evicts before they are complete.
template <int NB, int R, bool WIDE = false, int KB = 8>
__device__ __forceinline__ uint32_t decode_symbols(DecState &st, const uint16_t *table, int32_t C,
                                                   int32_t N, float a, const float *deq,
                                                   uint16_t *orow, uint32_t one)
{
    static_assert(KB == 8 || KB == 16, "8 or 16 symbols per store");
    const int32_t Lp = N + 1;
    uint32_t x = st.x, d = st.d, v = st.v;
    Bits br = st.br;
    const uint32_t top_step = 1u << (31 - __clz((uint32_t)(N - 1)));
    uint32_t short_batch = 0;
    // the next word of the stream, loaded one refill ahead
    uint32_t nw = 0;
    if (R > 1)
        nw = *reinterpret_cast<const uint32_t *>(br.base + min(br.pos, br.lim));
    // shared addresses: r32 of the current symbol's CDF row, and kq with
    // kq + 2 p = the dequantisation entry of the symbol whose lower bound
    // sits at address p of that row
    const uint32_t tab32 = smem_u32(table);
    uint32_t r32 = tab32;
    uint32_t kq = smem_u32(deq) - 2u * tab32;

    // one symbol (j: its place in the block, for the refill cadence);
    // returns its dequantised value
    auto symbol = [&](int j) -> float {
        // the largest s with floor(r * cdf[s] / 2^16) <= v (the coder's own
        // comparison, so the result is exact); p = the address of cdf[s]
        uint32_t p = r32;
        const uint32_t T = search_target(d, v);
        if (NB == 16) {
            search_4way(p, 4, T, one);
            if (WIDE) {
                search_4way(p, 1, T, one);
            } else {
                search_2way(p, 2, T, one);
                search_2way(p, 1, T, one);
            }
        } else if (NB == 32) {
            search_4way(p, 8, T, one);
            search_4way(p, 2, T, one);
            search_2way(p, 1, T, one);
        } else {
            for (uint32_t step = top_step; step != 0; step >>= 1) {
                const uint32_t t = p + 2 * step;
                if (t - r32 < 2 * (uint32_t)N && lds_u16(t) <= T)
                    p = t;
            }
        }
        // s <= N - 1, so both bounds lie in the row. A valid stream never
        // holds the top symbol N - 1 (never coded); a corrupt one that reaches
        // it gets cdf[N] (stored as 0) as its upper bound and decodes to
        // garbage, still inside the buffers.
        uint32_t t0 = scale16(d, lds_u16(p));
        uint32_t dn = scale16(d, lds_u16(p + 2)) - t0 - 1u;
        if (v - t0 > dn) {
            // the target missed a bound (rare): search with the exact compare
            const char *rb = reinterpret_cast<const char *>(table) + (r32 - tab32);
            p = r32 + exact_search<NB>(rb, d, v, N, top_step);
            t0 = scale16(d, lds_u16(p));
            dn = scale16(d, lds_u16(p + 2)) - t0 - 1u;
        }
        // renormalise (see Enc); v takes S new bits
        const uint32_t xs = x + t0;
        const uint32_t S = renorm_shift(xs, dn);
        x = shl_clamped(xs, S);
        d = __funnelshift_l(0xFFFFFFFFu, dn, S);
        v = __funnelshift_l(br.b1, v - t0, S);
        if (R == 1) {
            bits_skip(br, S);
        } else {
            br.b1 = __funnelshift_l(br.b0, br.b1, S);
            br.b0 = shl_clamped(br.b0, S);
            br.avail -= (int32_t)S;
            if ((j % R) == R - 1) {
                short_batch |= (br.avail < 0) ? 1u : 0u;
                bits_refill_next(br, nw);
            }
        }
        // dequantise: fp32((q - MAX) / MAX) * a, entry s of deq (4 bytes
        // per entry, 2 per CDF entry)
        const uint32_t qa = kq + 2u * p;
        r32 += 2 * Lp;
        kq -= 4 * Lp;
        return __fmul_rn(lds_f32(qa), a);
    };
    // two values per bf16 conversion (each rounded to nearest even on its own)
    auto pack = [](float lo, float hi) -> uint32_t {
        const __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&pr);
    };

    // the output is written once and not read here: its stores allocate no
    // L1 line and take an L2 evict-first policy, so that the 2 GiB streaming
    // out of a large call leave the bit-stream words in L1 and L2
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    for (int32_t c0 = 0; c0 < C; c0 += KB) {
        uint32_t p[KB / 2];
#pragma unroll
        for (int j = 0; j < KB; j += 2) {
            const float lo = symbol(j);
            p[j >> 1] = pack(lo, symbol(j + 1));
        }
        if (KB == 16)
            asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], "
                         "{%1, %2, %3, %4, %5, %6, %7, %8}, %9;"
                         :
                         : "l"(orow + c0), "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]),
                           "r"(p[4 % (KB / 2)]), "r"(p[5 % (KB / 2)]), "r"(p[6 % (KB / 2)]),
                           "r"(p[7 % (KB / 2)]), "l"(pol)
                         : "memory");
        else
            asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                         :
                         : "l"(orow + c0), "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "l"(pol)
                         : "memory");
    }
    st.x = x;
    st.d = d;
    st.v = v;
    st.br = br;
#ifdef CG_TEST_EXACT_PATHS
    if (R > 1)
        short_batch = 1;
#endif
    return short_batch;
}

// Decode one stream (C symbols) and write its dequantised row. R > 1
// refills the bit buffer once per R symbols and returns 1 when a batch ran
// short of bits (the output is then wrong and the caller decodes the stream
// again with R = 1, which never runs short: a symbol takes at most 18 bits
// and the buffer holds at least 33 after every refill).
template <int NB, int R, bool WIDE = false, int KB = 8>
__device__ __forceinline__ uint32_t decode_stream(const uint16_t *table, int32_t C, int32_t N,
                                                  const Bits &br, float a, const float *deq,
                                                  uint16_t *orow, uint32_t one)
{
    DecState st;
    dec_start(st, br);
    return decode_symbols<NB, R, WIDE, KB>(st, table, C, N, a, deq, orow, one);
}

// The refill-per-symbol decode of one stream, out of line: it runs only for
// streams whose batched decode ran short of bits.
template <int NB>
__device__ __noinline__ void decode_stream_exact(const uint16_t *table, int32_t C, int32_t N,
                                                 const uint8_t *bytestream, uint64_t sb,
                                                 uint64_t last, float a, const float *deq,
                                                 uint16_t *orow, uint32_t one)
{
    Bits br;
    bits_init(br, bytestream, sb, last);
    decode_stream<NB, 1>(table, C, N, br, a, deq, orow, one);
}

// The same for the symbols of one channel part, from the state `st` held
// at the part's start (updated to the state after the part).
template <int NB>
__device__ __noinline__ void decode_part_exact(DecState *st, const uint16_t *table, int32_t C,
                                               int32_t N, float a, const float *deq,
                                               uint16_t *orow, uint32_t one)
{
    DecState s = *st;
    decode_symbols<NB, 1>(s, table, C, N, a, deq, orow, one);
    *st = s;
}

// One tile of the decoder; NB as in encode_tile. The CTA takes streams
// [h * NTH, (h + 1) * NTH) of the tile; KB as in decode_symbols.
template <int NB, int NTH, int KB>
__device__ __forceinline__ void decode_tile(const Tile &tl, const cg_tile_params &P,
                                            const uint8_t *__restrict__ bytestream,
                                            uint64_t stream_bytes,
                                            const int32_t *__restrict__ lengths,
                                            const uint16_t *__restrict__ cdf,
                                            const float *__restrict__ amax,
                                            const uint64_t *__restrict__ tile_base,
                                            uint16_t *__restrict__ kv_out,
                                            uint32_t *__restrict__ status, uint8_t *smem,
                                            uint32_t *warp_sums, float *deq, uint32_t *bad,
                                            int32_t h, uint32_t *offs, uint64_t *bar)
{
    const int32_t C = P.C;
    const int32_t N = NB > 0 ? NB : tl.N;
    const int32_t Lp = N + 1;
    const int32_t M = N / 2 - 1;
    const int tid = threadIdx.x;
    const int32_t sidx = h * NTH + tid;
    uint16_t *table = reinterpret_cast<uint16_t *>(smem);

    if (tid == 0) {
        *bad = 0;
        mbar_init(bar);
    }
    __syncthreads();
    // the table's bulk copy runs while the lengths are scanned
    const bool bulk = stage_table<NTH>(table, cdf + tl.cdf_base, (uint32_t)C * Lp * 2u, bar);
    if (tid < N)
        deq[tid] = __fdiv_rn((float)(tid - M), (float)M);
    uint32_t len = 0;
    const uint32_t off = tile_stream_offset<NTH>(tl, lengths, h, &len, warp_sums, offs);
    if (bulk && !mbar_wait(bar, 0))
        *bad = 2;
    // every row must start at 0, rise strictly and end at 65536 (stored 0)
    for (int32_t c = tid; c < C; c += NTH) {
        const uint16_t *row = table + (size_t)c * Lp;
        uint32_t ok = (row[0] == 0) && (row[N] == 0);
        for (int32_t i = 1; i < N; ++i)
            ok &= (row[i] > row[i - 1]) ? 1u : 0u;
        if (!ok)
            atomicMax(bad, 1u);
    }
    __syncthreads();
    if (*bad) {
        if (tid == 0)
            set_status(status, *bad == 2 ? CG_ERR_TIMEOUT : CG_ERR_CORRUPT);
        if (*bad == 2)
            mbar_wait(bar, 0);  // one more bounded wait for the copy in flight
        return;
    }
    if (sidx >= tl.n)
        return;

    // the buffer holds stream_bytes (>= 1) bytes, rounded up to 16 (checked
    // by the host): its last whole word starts at round4(stream_bytes) - 4
    const uint64_t last = ((stream_bytes + 3) & ~(uint64_t)3) - 4;
    uint64_t sb = tile_base[tl.index] + off;
    if (sb + len > stream_bytes) {
        set_status(status, CG_ERR_CORRUPT);
        sb = min(sb, last);
    }
    const float a = amax[((size_t)tl.kv * P.L + tl.l) * P.T + tl.t0 + sidx];
    uint16_t *orow = kv_out + ((size_t)(tl.l * 2 + tl.kv) * P.T + tl.t0 + sidx) * (size_t)C;
    Bits br;
    bits_init(br, bytestream, sb, last);
    if (decode_stream<NB, kRefillEvery, (NTH < NT), KB>(table, C, N, br, a, deq, orow, P.one))
        decode_stream_exact<NB>(table, C, N, bytestream, sb, last, a, deq, orow, P.one);
}

// One tile of the decoder whose CDF table is staged in channel parts of
// part_ch channels (a multiple of 8): tables too large for several CTAs per
// SM (32 and 64 bins at 1024 channels, 16 bins at 4096) take the shared
// memory of one part. Every stream decodes a part's channels, its coder state
// staying in registers; a block barrier separates the parts. A stream whose
// batched decode of a part ran short of bits decodes that part again, from
// the state it held at the part's start, refilling after every symbol.
template <int NB, int NTH, int KB>
__device__ __forceinline__ void decode_tile_parts(const Tile &tl, const cg_tile_params &P,
                                                  const uint8_t *__restrict__ bytestream,
                                                  uint64_t stream_bytes,
                                                  const int32_t *__restrict__ lengths,
                                                  const uint16_t *__restrict__ cdf,
                                                  const float *__restrict__ amax,
                                                  const uint64_t *__restrict__ tile_base,
                                                  uint16_t *__restrict__ kv_out,
                                                  uint32_t *__restrict__ status, uint8_t *smem,
                                                  uint32_t *warp_sums, float *deq, uint32_t *bad,
                                                  int32_t part_ch, int32_t h, uint32_t *offs,
                                                  uint64_t *bar)
{
    const int32_t C = P.C;
    const int32_t N = NB > 0 ? NB : tl.N;
    const int32_t Lp = N + 1;
    const int32_t M = N / 2 - 1;
    const int tid = threadIdx.x;
    const int32_t sidx = h * NTH + tid;
    uint16_t *table = reinterpret_cast<uint16_t *>(smem);

    if (tid == 0) {
        *bad = 0;
        mbar_init(bar);
    }
    __syncthreads();
    // the first part's bulk copy runs while the lengths are scanned
    bool bulk = stage_table<NTH>(table, cdf + tl.cdf_base, (uint32_t)min(part_ch, C) * Lp * 2u, bar);
    if (tid < N)
        deq[tid] = __fdiv_rn((float)(tid - M), (float)M);
    uint32_t len = 0;
    const bool active = sidx < tl.n;
    const uint32_t off = tile_stream_offset<NTH>(tl, lengths, h, &len, warp_sums, offs);
    DecState st;
    float a = 0.0f;
    uint16_t *orow = kv_out;
    if (active) {
        const uint64_t last = ((stream_bytes + 3) & ~(uint64_t)3) - 4;
        uint64_t sb = tile_base[tl.index] + off;
        if (sb + len > stream_bytes) {
            set_status(status, CG_ERR_CORRUPT);
            sb = min(sb, last);
        }
        a = amax[((size_t)tl.kv * P.L + tl.l) * P.T + tl.t0 + sidx];
        orow = kv_out + ((size_t)(tl.l * 2 + tl.kv) * P.T + tl.t0 + sidx) * (size_t)C;
        Bits br;
        bits_init(br, bytestream, sb, last);
        dec_start(st, br);
    }
    uint32_t phase = 0;
    for (int32_t c_begin = 0; c_begin < C; c_begin += part_ch, phase ^= 1u) {
        const int32_t nch = min(part_ch, C - c_begin);
        if (c_begin > 0)  // after the block barrier that ends the previous part
            bulk = stage_table<NTH>(table, cdf + tl.cdf_base + (size_t)c_begin * Lp,
                                    (uint32_t)nch * Lp * 2u, bar);
        if (bulk) {
            if (!mbar_wait(bar, phase))
                *bad = 2;
        } else {
            __syncthreads();  // the plain copy is complete
        }
        for (int32_t c = tid; c < nch; c += NTH) {
            const uint16_t *row = table + (size_t)c * Lp;
            uint32_t ok = (row[0] == 0) && (row[N] == 0);
            for (int32_t i = 1; i < N; ++i)
                ok &= (row[i] > row[i - 1]) ? 1u : 0u;
            if (!ok)
                atomicMax(bad, 1u);
        }
        __syncthreads();
        if (*bad) {
            if (tid == 0)
                set_status(status, *bad == 2 ? CG_ERR_TIMEOUT : CG_ERR_CORRUPT);
            if (*bad == 2)
                mbar_wait(bar, phase);  // one more bounded wait for the copy in flight
            return;
        }
        if (active) {
            const DecState saved = st;
            if (decode_symbols<NB, kRefillEvery, (NTH < NT), KB>(st, table, nch, N, a, deq,
                                                                 orow + c_begin, P.one)) {
                st = saved;
                decode_part_exact<NB>(&st, table, nch, N, a, deq, orow + c_begin, P.one);
            }
        }
        __syncthreads();  // the next part overwrites the table
    }
}

// Decoder tiles of one launch class (NB bins; 0 = any), at least MINB
// 256-thread CTAs' worth per SM; PARTS: the CDF table is staged in parts of
// part_ch channels; NTH < 256: each tile's streams are split over 256 / NTH
// CTAs of NTH threads (for calls with too few tiles to fill the GPU); KB:
// symbols per output store (decode_symbols).
template <int NB, int MINB, bool PARTS, int NTH, int KB = 8>
__global__ void __launch_bounds__(NTH, MINB *(NT / NTH))
    k_decode_class(const cg_tile_params P, int32_t cls_begin,
                   const uint8_t *__restrict__ bytestream, uint64_t stream_bytes,
                   const int32_t *__restrict__ lengths, const uint16_t *__restrict__ cdf,
                   const float *__restrict__ amax, const uint64_t *__restrict__ tile_base,
                   uint16_t *__restrict__ kv_out, uint32_t *__restrict__ status, int32_t part_ch)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t warp_sums[NTH / 32];
    __shared__ float deq[64];
    __shared__ uint32_t bad;
    __shared__ uint32_t offs[NTH < NT ? NT : 1];
    __shared__ uint64_t bar;
    constexpr int split = NT / NTH;
    const Tile tl = tile_of_class(P, cls_begin, blockIdx.x / split);
    const int32_t h = (int32_t)(blockIdx.x % split);
    if (PARTS)
        decode_tile_parts<NB, NTH, KB>(tl, P, bytestream, stream_bytes, lengths, cdf, amax, tile_base,
                                   kv_out, status, smem, warp_sums, deq, &bad, part_ch, h, offs,
                                   &bar);
    else
        decode_tile<NB, NTH, KB>(tl, P, bytestream, stream_bytes, lengths, cdf, amax, tile_base,
                             kv_out, status, smem, warp_sums, deq, &bad, h, offs, &bar);
}

// The kernel of each class, by bin count: 16 and 32 have specialised
// bodies and their own register budgets.
typedef void (*encode_fn)(const uint16_t *, const cg_tile_params, int32_t, uint8_t *, float *,
                          uint16_t *, int32_t *, uint8_t *, uint32_t *, uint32_t *, int32_t);
typedef void (*decode_fn)(const cg_tile_params, int32_t, const uint8_t *, uint64_t,
                          const int32_t *, const uint16_t *, const float *, const uint64_t *,
                          uint16_t *, uint32_t *, int32_t);

encode_fn encode_kernel(int32_t bins, bool parts, bool groups)
{
    if (bins == 16)
        return parts    ? k_encode_class<16, 4, true, false>
               : groups ? k_encode_class<16, 4, false, true>
                        : k_encode_class<16, 4, false, false>;
    if (bins == 32)
        return parts    ? k_encode_class<32, 4, true, false>
               : groups ? k_encode_class<32, 3, false, true>
                        : k_encode_class<32, 3, false, false>;
    return parts    ? k_encode_class<0, 4, true, false>
           : groups ? k_encode_class<0, 3, false, true>
                    : k_encode_class<0, 3, false, false>;
}

// whether a class of `bins` bins counts by row groups at C channels
bool encode_groups(int32_t C, int32_t bins)
{
    int32_t w = 0, r = 1;
    cg_count_layout(C, bins, &w, &r);
    return r > 1;
}

template <int NTH, int KB>
decode_fn decode_kernel_nth(int32_t bins, bool parts)
{
    if (bins == 16)
        return parts ? k_decode_class<16, 4, true, NTH, KB>
                     : k_decode_class<16, (NTH == NT ? 6 : 4), false, NTH, KB>;
    if (bins == 32)
        return parts ? k_decode_class<32, 4, true, NTH, KB> : k_decode_class<32, 3, false, NTH, KB>;
    return parts ? k_decode_class<0, 4, true, NTH, KB> : k_decode_class<0, 3, false, NTH, KB>;
}

// split: CTAs per tile (1, 2 or 4); sectors: every row (or row part) the
// launch writes is a whole number of 32-byte sectors at a 32-byte aligned
// address, for 32-byte output stores (one CTA per tile only: the split
// kernels, for small calls, keep 16-byte stores)
decode_fn decode_kernel(int32_t bins, bool parts, int split, bool sectors)
{
    if (split == 4)
        return decode_kernel_nth<NT / 4, 8>(bins, parts);
    if (split == 2)
        return decode_kernel_nth<NT / 2, 8>(bins, parts);
    return sectors ? decode_kernel_nth<NT, 16>(bins, parts) : decode_kernel_nth<NT, 8>(bins, parts);
}

// Number of SMs of the current device.
cudaError_t sm_count(int *sms)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess)
        err = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    return err;
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
    const int32_t bins[3] = {16, 32, 0};
    for (int i = 0; i < 3 && err == cudaSuccess; ++i) {
        // the plan keeps dynamic shared memory below CG_SMEM_LIMIT - 2048,
        // which leaves room for the kernels' static shared memory
        for (int v = 0; v < 3 && err == cudaSuccess; ++v)
            err = cudaFuncSetAttribute(encode_kernel(bins[i], v == 1, v == 2),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       CG_SMEM_LIMIT - 2048);
        for (int parts = 0; parts < 2 && err == cudaSuccess; ++parts)
            for (int split = 1; split <= 4 && err == cudaSuccess; split *= 2)
                for (int sectors = 0; sectors < 2 && err == cudaSuccess; ++sectors)
                    err = cudaFuncSetAttribute(decode_kernel(bins[i], parts != 0, split, sectors != 0),
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               CG_SMEM_LIMIT - 2048);
    }
    if (err == cudaSuccess)
        done.fetch_or(bit);
    return err;
}

}  // namespace

int32_t cg_encode_part_channels(int32_t C, int32_t bins)
{
    const size_t table = (size_t)C * (bins + 1) * 2;
    if (C < 4 * CG_TILE_THREADS || C % 32 != 0 || table <= CG_DECODE_TABLE_BUDGET)
        return C;
    const int32_t parts = (int32_t)((table + CG_DECODE_TABLE_BUDGET - 1) / CG_DECODE_TABLE_BUDGET);
    return ((C + parts - 1) / parts + 31) / 32 * 32;
}

size_t cg_smem_encode(int32_t C, int32_t bins)
{
    const size_t ch = (size_t)cg_encode_part_channels(C, bins);
    int32_t w = 0, r = 1;
    if (ch == (size_t)C)
        cg_count_layout(C, bins, &w, &r);
    return (((size_t)r * ch * (bins + 1) * 2 + 15) & ~(size_t)15) + CG_GROUP_TOKENS * sizeof(float);
}

int32_t cg_decode_part_channels(int32_t C, int32_t bins)
{
    const size_t table = (size_t)C * (bins + 1) * 2;
    if (table <= CG_DECODE_TABLE_BUDGET)
        return C;
    const int32_t parts = (int32_t)((table + CG_DECODE_TABLE_BUDGET - 1) / CG_DECODE_TABLE_BUDGET);
    return ((C + parts - 1) / parts + 7) / 8 * 8;
}

size_t cg_smem_decode(int32_t C, int32_t bins)
{
    return ((size_t)cg_decode_part_channels(C, bins) * (bins + 1) * 2 + 15) & ~(size_t)15;
}

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

int cg_encode_launch_count(const cg_plan *p) { return (int)p->classes.size() + 2; }
int cg_decode_launch_count(const cg_plan *p) { return (int)p->classes.size() + 2; }

cudaError_t cg_side_stream::ensure()
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (stream != nullptr && device == dev)
        return cudaSuccess;
    release();
    err = cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
    if (err == cudaSuccess) {
        int least = 0, greatest = 0;
        err = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (err == cudaSuccess)
            err = cudaStreamCreateWithPriority(&stream_hi, cudaStreamNonBlocking, greatest);
    }
    if (err == cudaSuccess)
        err = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    if (err == cudaSuccess)
        err = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        release();
        return err;
    }
    device = dev;
    return cudaSuccess;
}

void cg_side_stream::release()
{
    if (stream)
        cudaStreamDestroy(stream);
    if (stream_hi)
        cudaStreamDestroy(stream_hi);
    if (fork)
        cudaEventDestroy(fork);
    if (join)
        cudaEventDestroy(join);
    stream = stream_hi = nullptr;
    fork = join = nullptr;
    device = -1;
}

namespace {

// Launch every class: the class with the most tiles on the caller's stream,
// the others on a side stream, forked after the work already enqueued and
// joined back before anything enqueued later. With `first`, the side
// stream is the one at the greatest priority, so the block scheduler
// dispatches all of those classes' tiles before the main class's: the
// encoder's 32-bin tiles take longer than its 16-bin ones, and the short
// tiles then fill the end of the call (encode 2.01 -> 1.94 ms at 16K
// tokens; the decoder, whose 32-bin tiles hold fewer warps per SM, does not
// gain).
template <typename F>
cudaError_t launch_classes(const cg_plan *p, cudaStream_t stream, F launch, bool first)
{
    if (p->classes.size() == 1) {
        launch(p->classes[0], stream);
        return cudaGetLastError();
    }
    cudaError_t err = p->side.ensure();
    if (err != cudaSuccess)
        return err;
    size_t main = 0;
    for (size_t i = 1; i < p->classes.size(); ++i)
        if (p->classes[i].count > p->classes[main].count)
            main = i;
    cudaStream_t side = first ? p->side.stream_hi : p->side.stream;
    err = cudaEventRecord(p->side.fork, stream);
    if (err == cudaSuccess)
        err = cudaStreamWaitEvent(side, p->side.fork, 0);
    if (err != cudaSuccess)
        return err;
    for (size_t i = 0; i < p->classes.size(); ++i)
        if (i != main)
            launch(p->classes[i], side);
    launch(p->classes[main], stream);
    err = cudaEventRecord(p->side.join, side);
    if (err == cudaSuccess)
        err = cudaStreamWaitEvent(stream, p->side.join, 0);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

}  // namespace

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
    err = launch_classes(p, stream, [&](const cg_bin_class &cl, cudaStream_t s) {
        const int32_t part_ch = cg_encode_part_channels(p->C, cl.bins);
        encode_kernel(cl.bins, part_ch < p->C, encode_groups(p->C, cl.bins))<<<
            p->tp.ngroups * cl.count, NT, cl.smem_encode, s>>>(
            static_cast<const uint16_t *>(kv), p->tp, cl.begin, sym, out->amax, out->cdf,
            out->lengths, slots, tile_totals, status, part_ch);
    }, true);
    p->prof.end(stream);
    if (err != cudaSuccess)
        return err;
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
    int sms = 0;
    err = sm_count(&sms);
    if (err != cudaSuccess)
        return err;
    // a call with fewer than 1.5 tiles per SM would leave some SMs with two
    // tiles and others with one (the launch then takes two tiles' time): it
    // splits each tile's streams over 4 CTAs of 64 threads, which spreads
    // evenly. With more tiles per SM the imbalance is small and the copies of
    // the CDF table that a split costs outweigh it.
    const int split = ((int64_t)ntiles * 2 < (int64_t)sms * 3) ? 4 : 1;
    err = launch_classes(p, stream, [&](const cg_bin_class &cl, cudaStream_t s) {
        const int32_t part_ch = cg_decode_part_channels(p->C, cl.bins);
        const bool sectors = p->C % 16 == 0 && part_ch % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(kv_out) % 32 == 0;
        decode_kernel(cl.bins, part_ch < p->C, split, sectors)<<<
            p->tp.ngroups * cl.count * split, NT / split, cl.smem_decode, s>>>(
            p->tp, cl.begin, in->bytestream, stream_bytes, in->lengths, in->cdf, in->amax,
            tile_base, static_cast<uint16_t *>(kv_out), status, part_ch);
    }, false);
    p->prof.end(stream);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}
