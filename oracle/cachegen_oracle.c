/*
 * CacheGen KV-cache codec: plain CPU oracle.
 *
 * TEST INFRASTRUCTURE. This is the slow, obviously-correct reference that
 * the CUDA path is checked against. Only the test-suite, the package's
 * smoke check and the bench's CPU-baseline leg load it; the product path
 * never does. It shares no code, header, table or helper with the CUDA
 * path. Build with `-ffp-contract=off` so that every float operation below
 * is rounded on its own, in the order written.
 *
 * Sources (cited by title and section):
 *   [CG-LMCache] "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与
 *                源码解析" (0539edu.com/news/4720135):
 *                §1 QuantizationSpec, §2 Quantization, §3 CDF estimation and
 *                normalisation, §4 arithmetic coding and GPU kernels,
 *                §5 decoding and dequantisation.
 *   [WNC87]      I. H. Witten, R. M. Neal, J. G. Cleary, "Arithmetic coding
 *                for data compression", CACM 30(6), 1987: the 32-bit
 *                low/high integer coder with pending (underflow) bits.
 *
 * Readings taken where the page is silent (each is listed in the design
 * notes): one scale per (K/V, layer, token) over channels; fp32 quantise
 * math as two separately rounded operations, ties to even; an all-zero row
 * gets factor 0; alphabet N = bins and a CDF of N+1 entries; the float CDF
 * is replaced by the exact integer floor(cum*(65536-N)/n) + i; one stream
 * per (K/V, layer, token) holding the C channels in order; streams ordered
 * group -> K/V -> layer -> token; MSB-first bits, zero padding, bits past a
 * stream's end read as 0.
 *
 * Layouts: kv is [L][2][T][C] bf16 bits (uint16) with C = heads*head_size;
 * amax is [2][L][T] fp32; symbols are [2][L][T][C] uint8; the wire CDF is
 * uint16, per group -> K/V -> layer -> channel -> N+1 entries, with 65536
 * stored as 0.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_INVALID_ARG 1
#define ORC_ERR_SPEC 2
#define ORC_ERR_CAPACITY 3
#define ORC_ERR_NONFINITE 4
#define ORC_ERR_CORRUPT 5

/* [CG-LMCache §4]: tokens are processed in batches of at most 256, each
 * batch with its own CDFs. */
#define ORC_GROUP_TOKENS 256

/* [CG-LMCache §3]: the integer CDF is scaled to 2^16. */
#define ORC_CDF_TOTAL 65536u

/* [WNC87] 32-bit code values. */
#define WNC_TOP 0xFFFFFFFFull
#define WNC_HALF 0x80000000ull
#define WNC_QUARTER 0x40000000ull
#define WNC_3QUARTER 0xC0000000ull

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                        */
/* ------------------------------------------------------------------ */

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even, keeping the top 16 bits. Inputs here are
 * always finite. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

/* ------------------------------------------------------------------ */
/* Configuration [CG-LMCache §1]                                        */
/* ------------------------------------------------------------------ */

/* Expand a list of {start_layer, end_layer, bins} triples (layer range
 * [start, end)) into one bin count per layer. The triples must cover
 * [0, L) exactly once; bins must be even and in [4, 64]. */
int orc_layer_bins(int32_t L, const int32_t *specs, int32_t nspecs, int32_t *bins)
{
    if (L <= 0 || nspecs <= 0 || specs == NULL || bins == NULL)
        return ORC_ERR_INVALID_ARG;
    for (int32_t l = 0; l < L; ++l)
        bins[l] = 0;
    for (int32_t i = 0; i < nspecs; ++i) {
        int32_t start = specs[3 * i + 0];
        int32_t end = specs[3 * i + 1];
        int32_t b = specs[3 * i + 2];
        if (start < 0 || end > L || start >= end)
            return ORC_ERR_SPEC;
        if (b < 4 || b > 64 || (b % 2) != 0)
            return ORC_ERR_SPEC;
        for (int32_t l = start; l < end; ++l) {
            if (bins[l] != 0)
                return ORC_ERR_SPEC; /* overlap */
            bins[l] = b;
        }
    }
    for (int32_t l = 0; l < L; ++l)
        if (bins[l] == 0)
            return ORC_ERR_SPEC; /* gap */
    return ORC_OK;
}

/* Token groups: the blob is cut into objects of chunk_tokens tokens (the
 * last may be short), and each object into runs of at most 256 tokens
 * [CG-LMCache §4]. Writes start/count for each group when the arrays are
 * given; returns the number of groups (or -1 on bad arguments). */
int32_t orc_groups(int32_t T, int32_t chunk_tokens, int32_t *start, int32_t *count)
{
    if (T <= 0 || chunk_tokens <= 0)
        return -1;
    int32_t g = 0;
    int32_t t = 0;
    while (t < T) {
        int32_t obj_end = (T - t > chunk_tokens) ? t + chunk_tokens : T;
        for (int32_t u = t; u < obj_end; u += ORC_GROUP_TOKENS) {
            int32_t n = obj_end - u;
            if (n > ORC_GROUP_TOKENS)
                n = ORC_GROUP_TOKENS;
            if (start)
                start[g] = u;
            if (count)
                count[g] = n;
            ++g;
        }
        t = obj_end;
    }
    return g;
}

/* ------------------------------------------------------------------ */
/* Quantisation [CG-LMCache §2]                                         */
/* ------------------------------------------------------------------ */

/* One row (one K/V, layer, token) of C channels.
 *   MAX = bins/2 - 1,  a = max_c |x_c|,  f = MAX / a,
 *   q_c = round(x_c * f + MAX)   (two fp32 roundings, ties to even).
 * An all-zero row (a == 0) takes f = 0, so every q is MAX. */
int orc_quantize_row(const uint16_t *x, int32_t C, int32_t bins, float *amax_out, uint8_t *q)
{
    int32_t M = bins / 2 - 1;
    float a = 0.0f;
    for (int32_t c = 0; c < C; ++c) {
        float v = fabsf(bf16_to_float(x[c]));
        if (!isfinite(v))
            return ORC_ERR_NONFINITE;
        if (v > a)
            a = v;
    }
    float f = (a == 0.0f) ? 0.0f : (float)M / a;
    /* Reading: a row so small that MAX / a overflows fp32 (a below about
     * 2^-124) has no finite scale factor; it is rejected like inf/NaN. */
    if (!isfinite(f))
        return ORC_ERR_NONFINITE;
    for (int32_t c = 0; c < C; ++c) {
        float y = bf16_to_float(x[c]) * f;
        y = y + (float)M;
        float r = rintf(y);
        int32_t iq = (int32_t)r;
        if (iq < 0 || iq > 2 * M)
            return ORC_ERR_INVALID_ARG; /* cannot happen for finite input */
        q[c] = (uint8_t)iq;
    }
    *amax_out = a;
    return ORC_OK;
}

/* Inverse scaling [CG-LMCache §5]: t = (q - MAX) / MAX * a, then cast back
 * to bf16 (round to nearest even). */
void orc_dequant_row(const uint8_t *q, int32_t C, int32_t bins, float a, uint16_t *y)
{
    int32_t M = bins / 2 - 1;
    float fm = (float)M;
    for (int32_t c = 0; c < C; ++c) {
        float t = (float)((int32_t)q[c] - M);
        t = t / fm;
        t = t * a;
        y[c] = float_to_bf16_rne(t);
    }
}

/* ------------------------------------------------------------------ */
/* Integer CDF [CG-LMCache §3]                                          */
/* ------------------------------------------------------------------ */

/* From a histogram of n symbols over an alphabet of N: the cumulative
 * count cum[i] (symbols < i), scaled by 2^16 - N with an exact floor, plus
 * the ramp i, so that cdf[0] = 0, cdf[N] = 65536 and every step is >= 1. */
void orc_int_cdf(const uint32_t *count, int32_t N, uint32_t n, uint32_t *cdf)
{
    uint64_t cum = 0;
    uint64_t scale = (uint64_t)ORC_CDF_TOTAL - (uint64_t)N;
    for (int32_t i = 0; i <= N; ++i) {
        cdf[i] = (uint32_t)((cum * scale) / n) + (uint32_t)i;
        if (i < N)
            cum += count[i];
    }
}

/* A CDF row is usable by the coder when it starts at 0, ends at 65536 and
 * rises strictly. */
static int cdf_row_valid(const uint32_t *cdf, int32_t N)
{
    if (cdf[0] != 0 || cdf[N] != ORC_CDF_TOTAL)
        return 0;
    for (int32_t i = 0; i < N; ++i)
        if (cdf[i + 1] <= cdf[i])
            return 0;
    return 1;
}

/* ------------------------------------------------------------------ */
/* Arithmetic coder [WNC87]                                             */
/* ------------------------------------------------------------------ */

typedef struct {
    uint8_t *out;
    size_t cap;   /* bytes */
    size_t nbits; /* bits written */
    int overflow;
} bit_writer;

static void put_bit(bit_writer *w, int b)
{
    size_t byte = w->nbits >> 3;
    if (byte >= w->cap) {
        w->overflow = 1;
        w->nbits++;
        return;
    }
    if ((w->nbits & 7u) == 0)
        w->out[byte] = 0;
    if (b)
        w->out[byte] |= (uint8_t)(0x80u >> (w->nbits & 7u));
    w->nbits++;
}

/* Emit one bit, then the pending bits as its complement. */
static void put_bit_and_pending(bit_writer *w, int b, uint64_t *pending)
{
    put_bit(w, b);
    while (*pending > 0) {
        put_bit(w, !b);
        --*pending;
    }
}

/* Encode nsym symbols; symbol i uses CDF row cdf + i*row_stride (N+1
 * entries, 0..65536). For each symbol s with r = high - low + 1:
 *     high = low + floor(r*cdf[s+1] / 2^16) - 1,
 *     low  = low + floor(r*cdf[s]   / 2^16),
 * then renormalise: while the interval lies in the lower half, the upper
 * half or the middle half, emit 0 / emit 1 / count a pending bit, and
 * double. Termination: one more pending bit, then 0 if low < 1/4 else 1,
 * followed by the pending bits. Bits are packed MSB-first; the last byte
 * is zero-padded. *nbytes gets the stream length in bytes. */
int orc_wnc_encode(const uint8_t *sym, int32_t nsym, const uint32_t *cdf, int32_t row_stride,
                   int32_t N, uint8_t *out, size_t cap, size_t *nbytes)
{
    bit_writer w = {out, cap, 0, 0};
    uint64_t low = 0, high = WNC_TOP, pending = 0;
    for (int32_t i = 0; i < nsym; ++i) {
        const uint32_t *row = cdf + (size_t)i * (size_t)row_stride;
        int32_t s = sym[i];
        if (s >= N)
            return ORC_ERR_INVALID_ARG;
        uint64_t r = high - low + 1;
        high = low + ((r * row[s + 1]) >> 16) - 1;
        low = low + ((r * row[s]) >> 16);
        for (;;) {
            if (high < WNC_HALF) {
                put_bit_and_pending(&w, 0, &pending);
            } else if (low >= WNC_HALF) {
                put_bit_and_pending(&w, 1, &pending);
                low -= WNC_HALF;
                high -= WNC_HALF;
            } else if (low >= WNC_QUARTER && high < WNC_3QUARTER) {
                pending++;
                low -= WNC_QUARTER;
                high -= WNC_QUARTER;
            } else {
                break;
            }
            low = 2 * low;
            high = 2 * high + 1;
        }
    }
    pending++;
    if (low < WNC_QUARTER)
        put_bit_and_pending(&w, 0, &pending);
    else
        put_bit_and_pending(&w, 1, &pending);
    *nbytes = (w.nbits + 7) / 8;
    return w.overflow ? ORC_ERR_CAPACITY : ORC_OK;
}

typedef struct {
    const uint8_t *in;
    size_t nbits; /* stream length in bits */
    size_t pos;
} bit_reader;

/* Bits past the end of the stream read as 0. */
static uint64_t get_bit(bit_reader *r)
{
    uint64_t b = 0;
    if (r->pos < r->nbits)
        b = (r->in[r->pos >> 3] >> (7u - (r->pos & 7u))) & 1u;
    r->pos++;
    return b;
}

/* Decode nsym symbols from a stream of nbytes bytes with the same CDF rows
 * as the encoder. The symbol is the largest s whose sub-interval starts at
 * or below the code value; it is checked against the division form
 * floor(((value - low + 1) * 2^16 - 1) / r). */
int orc_wnc_decode(const uint8_t *in, size_t nbytes, int32_t nsym, const uint32_t *cdf,
                   int32_t row_stride, int32_t N, uint8_t *sym)
{
    bit_reader br = {in, nbytes * 8, 0};
    uint64_t low = 0, high = WNC_TOP, value = 0;
    for (int k = 0; k < 32; ++k)
        value = (value << 1) | get_bit(&br);
    for (int32_t i = 0; i < nsym; ++i) {
        const uint32_t *row = cdf + (size_t)i * (size_t)row_stride;
        uint64_t r = high - low + 1;
        int32_t s = 0;
        while (s + 1 < N && low + ((r * row[s + 1]) >> 16) <= value)
            ++s;
        uint64_t target = (((value - low + 1) << 16) - 1) / r;
        if (!(row[s] <= target && target < row[s + 1]))
            return ORC_ERR_CORRUPT;
        high = low + ((r * row[s + 1]) >> 16) - 1;
        low = low + ((r * row[s]) >> 16);
        for (;;) {
            if (high < WNC_HALF) {
                /* nothing to subtract */
            } else if (low >= WNC_HALF) {
                low -= WNC_HALF;
                high -= WNC_HALF;
                value -= WNC_HALF;
            } else if (low >= WNC_QUARTER && high < WNC_3QUARTER) {
                low -= WNC_QUARTER;
                high -= WNC_QUARTER;
                value -= WNC_QUARTER;
            } else {
                break;
            }
            low = 2 * low;
            high = 2 * high + 1;
            value = 2 * value + get_bit(&br);
        }
        sym[i] = (uint8_t)s;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Whole pipeline                                                       */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t L, T, C;
    int32_t ngroups;
    int32_t *gstart, *gcount;  /* [ngroups] */
    int32_t *bins;             /* [2][L] */
    size_t *cdf_off;           /* [ngroups][2][L] offset of the (g,kv,l) CDF block, entries */
    size_t cdf_entries;        /* total wire CDF entries */
} orc_layout;

static void layout_free(orc_layout *lo)
{
    free(lo->gstart);
    free(lo->gcount);
    free(lo->bins);
    free(lo->cdf_off);
    memset(lo, 0, sizeof *lo);
}

static int layout_make(orc_layout *lo, int32_t L, int32_t T, int32_t C, int32_t chunk_tokens,
                       const int32_t *kspecs, int32_t nk, const int32_t *vspecs, int32_t nv)
{
    memset(lo, 0, sizeof *lo);
    if (L <= 0 || T <= 0 || C <= 0 || chunk_tokens <= 0)
        return ORC_ERR_INVALID_ARG;
    lo->L = L;
    lo->T = T;
    lo->C = C;
    lo->bins = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)L);
    if (!lo->bins)
        return ORC_ERR_INVALID_ARG;
    int st = orc_layer_bins(L, kspecs, nk, lo->bins);
    if (st == ORC_OK)
        st = orc_layer_bins(L, vspecs, nv, lo->bins + L);
    if (st != ORC_OK) {
        layout_free(lo);
        return st;
    }
    lo->ngroups = orc_groups(T, chunk_tokens, NULL, NULL);
    lo->gstart = (int32_t *)malloc(sizeof(int32_t) * (size_t)lo->ngroups);
    lo->gcount = (int32_t *)malloc(sizeof(int32_t) * (size_t)lo->ngroups);
    lo->cdf_off = (size_t *)malloc(sizeof(size_t) * (size_t)lo->ngroups * 2 * (size_t)L);
    if (!lo->gstart || !lo->gcount || !lo->cdf_off) {
        layout_free(lo);
        return ORC_ERR_INVALID_ARG;
    }
    orc_groups(T, chunk_tokens, lo->gstart, lo->gcount);
    size_t off = 0;
    for (int32_t g = 0; g < lo->ngroups; ++g)
        for (int32_t kv = 0; kv < 2; ++kv)
            for (int32_t l = 0; l < L; ++l) {
                lo->cdf_off[((size_t)g * 2 + kv) * L + l] = off;
                off += (size_t)C * (size_t)(lo->bins[kv * L + l] + 1);
            }
    lo->cdf_entries = off;
    return ORC_OK;
}

/* Index of the first stream of tile (g, kv, l): streams are ordered group,
 * then K/V, then layer, then token within the group. */
static size_t tile_first_stream(const orc_layout *lo, int32_t g, int32_t kv, int32_t l)
{
    return (size_t)2 * lo->L * lo->gstart[g] + ((size_t)kv * lo->L + l) * lo->gcount[g];
}

int32_t orc_num_groups(int32_t T, int32_t chunk_tokens)
{
    return orc_groups(T, chunk_tokens, NULL, NULL);
}

/* Total wire CDF entries for a configuration (or -1 on a bad config). */
int64_t orc_cdf_entries(int32_t L, int32_t T, int32_t C, int32_t chunk_tokens, const int32_t *kspecs,
                        int32_t nk, const int32_t *vspecs, int32_t nv)
{
    orc_layout lo;
    if (layout_make(&lo, L, T, C, chunk_tokens, kspecs, nk, vspecs, nv) != ORC_OK)
        return -1;
    int64_t e = (int64_t)lo.cdf_entries;
    layout_free(&lo);
    return e;
}

/* Encode one tile: K/V kvsel, layer l, group g. Quantises the group's rows,
 * builds the per-channel histograms and integer CDFs, and codes one stream
 * per token. Outputs (all optional except out/lengths):
 *   amax[n], symbols[n*C], cdf_wire[C*(N+1)], lengths[n], out (streams
 *   concatenated, *used bytes). */
static int encode_tile(const orc_layout *lo, const uint16_t *kv, int32_t g, int32_t kvsel, int32_t l,
                       float *amax, uint8_t *symbols, uint16_t *cdf_wire, int32_t *lengths,
                       uint8_t *out, size_t cap, size_t *used)
{
    int32_t C = lo->C, T = lo->T;
    int32_t n = lo->gcount[g], t0 = lo->gstart[g];
    int32_t bins = lo->bins[kvsel * lo->L + l];
    int32_t N = bins;
    int32_t Lp = N + 1;
    int st = ORC_OK;
    uint8_t *q = (uint8_t *)malloc((size_t)n * C);
    uint32_t *count = (uint32_t *)calloc((size_t)C * N, sizeof(uint32_t));
    uint32_t *cdf = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)C * Lp);
    if (!q || !count || !cdf) {
        st = ORC_ERR_INVALID_ARG;
        goto done;
    }
    /* quantise */
    for (int32_t i = 0; i < n; ++i) {
        const uint16_t *row = kv + (((size_t)l * 2 + kvsel) * T + (size_t)(t0 + i)) * C;
        float a;
        st = orc_quantize_row(row, C, bins, &a, q + (size_t)i * C);
        if (st != ORC_OK)
            goto done;
        if (amax)
            amax[i] = a;
    }
    if (symbols)
        memcpy(symbols, q, (size_t)n * C);
    /* histogram over the group's tokens, per channel */
    for (int32_t i = 0; i < n; ++i)
        for (int32_t c = 0; c < C; ++c)
            count[(size_t)c * N + q[(size_t)i * C + c]]++;
    /* integer CDF per channel */
    for (int32_t c = 0; c < C; ++c) {
        orc_int_cdf(count + (size_t)c * N, N, (uint32_t)n, cdf + (size_t)c * Lp);
        if (!cdf_row_valid(cdf + (size_t)c * Lp, N)) {
            st = ORC_ERR_INVALID_ARG;
            goto done;
        }
    }
    if (cdf_wire)
        for (size_t e = 0; e < (size_t)C * Lp; ++e)
            cdf_wire[e] = (uint16_t)(cdf[e] & 0xFFFFu);
    /* one stream per token, channels in order */
    size_t pos = 0;
    for (int32_t i = 0; i < n; ++i) {
        size_t nb = 0;
        st = orc_wnc_encode(q + (size_t)i * C, C, cdf, Lp, N, out + pos, cap - pos, &nb);
        if (st != ORC_OK)
            goto done;
        lengths[i] = (int32_t)nb;
        pos += nb;
    }
    *used = pos;
done:
    free(q);
    free(count);
    free(cdf);
    return st;
}

/* Worst-case bytes of one stream: at most 16 bits per symbol (every
 * frequency is at least 1 of 2^16) plus the termination bits. */
static size_t stream_cap(int32_t C)
{
    return (size_t)2 * C + 2;
}

/* Encode a whole blob kv[L][2][T][C].
 * Outputs: amax[2][L][T]; cdf_wire (cdf_entries u16); lengths[2*L*T] in
 * stream order; bytes (capacity cap) with the streams concatenated in
 * stream order; *total = bytes used. symbols[2][L][T][C] is optional.
 * nthreads > 1 encodes tiles in parallel (OpenMP); the result does not
 * depend on it. */
int orc_encode(const uint16_t *kv, int32_t L, int32_t T, int32_t C, int32_t chunk_tokens,
               const int32_t *kspecs, int32_t nk, const int32_t *vspecs, int32_t nv, float *amax,
               uint16_t *cdf_wire, int32_t *lengths, uint8_t *bytes, size_t cap, size_t *total,
               uint8_t *symbols, int32_t nthreads)
{
    orc_layout lo;
    int st = layout_make(&lo, L, T, C, chunk_tokens, kspecs, nk, vspecs, nv);
    if (st != ORC_OK)
        return st;
    size_t ntiles = (size_t)lo.ngroups * 2 * L;
    size_t *tile_used = (size_t *)calloc(ntiles, sizeof(size_t));
    uint8_t **tile_buf = (uint8_t **)calloc(ntiles, sizeof(uint8_t *));
    int *tile_st = (int *)calloc(ntiles, sizeof(int));
    if (!tile_used || !tile_buf || !tile_st) {
        st = ORC_ERR_INVALID_ARG;
        goto done;
    }
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long long ti = 0; ti < (long long)ntiles; ++ti) {
        int32_t g = (int32_t)(ti / (2 * L));
        int32_t kvsel = (int32_t)((ti / L) % 2);
        int32_t l = (int32_t)(ti % L);
        int32_t n = lo.gcount[g];
        size_t first = tile_first_stream(&lo, g, kvsel, l);
        size_t tcap = (size_t)n * stream_cap(C);
        tile_buf[ti] = (uint8_t *)malloc(tcap);
        float *tam = (float *)malloc(sizeof(float) * (size_t)n);
        uint8_t *tsym = symbols ? (uint8_t *)malloc((size_t)n * C) : NULL;
        if (!tile_buf[ti] || !tam || (symbols && !tsym)) {
            tile_st[ti] = ORC_ERR_INVALID_ARG;
        } else {
            tile_st[ti] = encode_tile(&lo, kv, g, kvsel, l, tam, tsym, cdf_wire + lo.cdf_off[ti],
                                      lengths + first, tile_buf[ti], tcap, &tile_used[ti]);
            if (tile_st[ti] == ORC_OK) {
                for (int32_t i = 0; i < n; ++i) {
                    size_t t = (size_t)lo.gstart[g] + i;
                    amax[((size_t)kvsel * L + l) * T + t] = tam[i];
                    if (symbols)
                        memcpy(symbols + (((size_t)kvsel * L + l) * T + t) * C,
                               tsym + (size_t)i * C, (size_t)C);
                }
            }
        }
        free(tam);
        free(tsym);
    }
    {
        size_t pos = 0;
        for (size_t ti = 0; ti < ntiles; ++ti) {
            if (tile_st[ti] != ORC_OK) {
                st = tile_st[ti];
                goto done;
            }
            if (pos + tile_used[ti] > cap) {
                st = ORC_ERR_CAPACITY;
                goto done;
            }
            memcpy(bytes + pos, tile_buf[ti], tile_used[ti]);
            pos += tile_used[ti];
        }
        *total = pos;
    }
done:
    if (tile_buf)
        for (size_t ti = 0; ti < ntiles; ++ti)
            free(tile_buf[ti]);
    free(tile_buf);
    free(tile_used);
    free(tile_st);
    layout_free(&lo);
    return st;
}

/* Decode one tile into symbols[n*C] (optional) and the bf16 rows of
 * kv_out. Reads the tile's wire CDF block; rejects rows that are not a
 * valid CDF. */
static int decode_tile(const orc_layout *lo, const uint8_t *bytes, const size_t *offsets,
                       const int32_t *lengths, const uint16_t *cdf_wire, const float *amax,
                       int32_t g, int32_t kvsel, int32_t l, uint16_t *kv_out, uint8_t *symbols)
{
    int32_t C = lo->C, T = lo->T, L = lo->L;
    int32_t n = lo->gcount[g], t0 = lo->gstart[g];
    int32_t bins = lo->bins[kvsel * L + l];
    int32_t N = bins, Lp = N + 1;
    size_t ti = ((size_t)g * 2 + kvsel) * L + l;
    const uint16_t *wire = cdf_wire + lo->cdf_off[ti];
    int st = ORC_OK;
    uint32_t *cdf = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)C * Lp);
    uint8_t *q = (uint8_t *)malloc((size_t)C);
    if (!cdf || !q) {
        st = ORC_ERR_INVALID_ARG;
        goto done;
    }
    for (int32_t c = 0; c < C; ++c) {
        uint32_t *row = cdf + (size_t)c * Lp;
        for (int32_t i = 0; i <= N; ++i)
            row[i] = wire[(size_t)c * Lp + i];
        if (row[N] != 0) {
            st = ORC_ERR_CORRUPT;
            goto done;
        }
        row[N] = ORC_CDF_TOTAL;
        if (!cdf_row_valid(row, N)) {
            st = ORC_ERR_CORRUPT;
            goto done;
        }
    }
    size_t first = tile_first_stream(lo, g, kvsel, l);
    for (int32_t i = 0; i < n; ++i) {
        size_t si = first + i;
        st = orc_wnc_decode(bytes + offsets[si], (size_t)lengths[si], C, cdf, Lp, N, q);
        if (st != ORC_OK)
            goto done;
        size_t t = (size_t)t0 + i;
        float a = amax[((size_t)kvsel * L + l) * T + t];
        orc_dequant_row(q, C, bins, a, kv_out + (((size_t)l * 2 + kvsel) * T + t) * C);
        if (symbols)
            memcpy(symbols + (((size_t)kvsel * L + l) * T + t) * C, q, (size_t)C);
    }
done:
    free(cdf);
    free(q);
    return st;
}

/* Decode a whole blob from the encoder's outputs into kv_out[L][2][T][C]
 * (bf16 bits). Stream offsets are the exclusive prefix sum of the lengths.
 * symbols[2][L][T][C] is optional. */
int orc_decode(const uint8_t *bytes, size_t nbytes, const int32_t *lengths, const uint16_t *cdf_wire,
               const float *amax, int32_t L, int32_t T, int32_t C, int32_t chunk_tokens,
               const int32_t *kspecs, int32_t nk, const int32_t *vspecs, int32_t nv,
               uint16_t *kv_out, uint8_t *symbols, int32_t nthreads)
{
    orc_layout lo;
    int st = layout_make(&lo, L, T, C, chunk_tokens, kspecs, nk, vspecs, nv);
    if (st != ORC_OK)
        return st;
    size_t S = (size_t)2 * L * T;
    size_t ntiles = (size_t)lo.ngroups * 2 * L;
    size_t *offsets = (size_t *)malloc(sizeof(size_t) * S);
    int *tile_st = (int *)calloc(ntiles, sizeof(int));
    if (!offsets || !tile_st) {
        st = ORC_ERR_INVALID_ARG;
        goto done;
    }
    {
        size_t pos = 0;
        for (size_t s = 0; s < S; ++s) {
            if (lengths[s] < 0) {
                st = ORC_ERR_CORRUPT;
                goto done;
            }
            offsets[s] = pos;
            pos += (size_t)lengths[s];
        }
        if (pos > nbytes) {
            st = ORC_ERR_CORRUPT;
            goto done;
        }
    }
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long long ti = 0; ti < (long long)ntiles; ++ti) {
        int32_t g = (int32_t)(ti / (2 * L));
        int32_t kvsel = (int32_t)((ti / L) % 2);
        int32_t l = (int32_t)(ti % L);
        tile_st[ti] = decode_tile(&lo, bytes, offsets, lengths, cdf_wire, amax, g, kvsel, l, kv_out,
                                  symbols);
    }
    for (size_t ti = 0; ti < ntiles; ++ti)
        if (tile_st[ti] != ORC_OK) {
            st = tile_st[ti];
            break;
        }
done:
    free(offsets);
    free(tile_st);
    layout_free(&lo);
    return st;
}

/* Encode a selection of tiles only (for sampled checks at sizes where the
 * whole blob is too slow). For each requested tile index ti (in
 * group -> K/V -> layer order) writes amax[n], cdf_wire[C*(N+1)],
 * lengths[n] and the tile's concatenated streams, packed one tile after
 * another in the output arrays; tile_bytes[k] gets the stream bytes of the
 * k-th requested tile. */
int orc_encode_tiles(const uint16_t *kv, int32_t L, int32_t T, int32_t C, int32_t chunk_tokens,
                     const int32_t *kspecs, int32_t nk, const int32_t *vspecs, int32_t nv,
                     const int64_t *tiles, int32_t ntiles_req, float *amax, uint16_t *cdf_wire,
                     int32_t *lengths, uint8_t *bytes, size_t cap, int64_t *tile_bytes,
                     int32_t nthreads)
{
    orc_layout lo;
    int st = layout_make(&lo, L, T, C, chunk_tokens, kspecs, nk, vspecs, nv);
    if (st != ORC_OK)
        return st;
    size_t ntiles = (size_t)lo.ngroups * 2 * L;
    size_t *tok_off = (size_t *)malloc(sizeof(size_t) * ((size_t)ntiles_req + 1));
    size_t *cdf_off = (size_t *)malloc(sizeof(size_t) * ((size_t)ntiles_req + 1));
    size_t *byte_off = (size_t *)malloc(sizeof(size_t) * ((size_t)ntiles_req + 1));
    int *tst = (int *)calloc((size_t)ntiles_req + 1, sizeof(int));
    if (!tok_off || !cdf_off || !byte_off || !tst) {
        st = ORC_ERR_INVALID_ARG;
        goto done;
    }
    tok_off[0] = cdf_off[0] = byte_off[0] = 0;
    for (int32_t k = 0; k < ntiles_req; ++k) {
        if (tiles[k] < 0 || (size_t)tiles[k] >= ntiles) {
            st = ORC_ERR_INVALID_ARG;
            goto done;
        }
        int32_t g = (int32_t)(tiles[k] / (2 * L));
        int32_t kvsel = (int32_t)((tiles[k] / L) % 2);
        int32_t l = (int32_t)(tiles[k] % L);
        int32_t n = lo.gcount[g];
        tok_off[k + 1] = tok_off[k] + (size_t)n;
        cdf_off[k + 1] = cdf_off[k] + (size_t)C * (lo.bins[kvsel * L + l] + 1);
        byte_off[k + 1] = byte_off[k] + (size_t)n * stream_cap(C);
    }
    if (byte_off[ntiles_req] > cap) {
        st = ORC_ERR_CAPACITY;
        goto done;
    }
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int32_t k = 0; k < ntiles_req; ++k) {
        int32_t g = (int32_t)(tiles[k] / (2 * L));
        int32_t kvsel = (int32_t)((tiles[k] / L) % 2);
        int32_t l = (int32_t)(tiles[k] % L);
        size_t used = 0;
        tst[k] = encode_tile(&lo, kv, g, kvsel, l, amax + tok_off[k], NULL, cdf_wire + cdf_off[k],
                             lengths + tok_off[k], bytes + byte_off[k],
                             byte_off[k + 1] - byte_off[k], &used);
        tile_bytes[k] = (int64_t)used;
    }
    for (int32_t k = 0; k < ntiles_req; ++k)
        if (tst[k] != ORC_OK) {
            st = tst[k];
            break;
        }
done:
    free(tok_off);
    free(cdf_off);
    free(byte_off);
    free(tst);
    layout_free(&lo);
    return st;
}

/* ------------------------------------------------------------------ */
/* Container                                                            */
/* ------------------------------------------------------------------ */

/* Flat little-endian container (version 1):
 *   "CGKV", u32 version, i32 L, T, heads, head_size, chunk_tokens,
 *   i32 n_kspecs, n_vspecs, i32 ngroups, u64 stream_bytes,          (48 B)
 *   specs: (n_kspecs + n_vspecs) x {i32 start, end, bins}, K first,
 *   amax f32[2][L][T], lengths i32[2*L*T], cdf u16[entries],
 *   streams u8[stream_bytes].
 * Returns the container size for the given sizes. */
int64_t orc_container_size(int32_t L, int32_t T, int32_t nspecs_total, int64_t cdf_entries,
                           int64_t stream_bytes)
{
    return 48 + (int64_t)12 * nspecs_total + (int64_t)4 * 2 * L * T + (int64_t)4 * 2 * L * T +
           (int64_t)2 * cdf_entries + stream_bytes;
}

static void put_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

int orc_serialize(int32_t L, int32_t T, int32_t H, int32_t D, int32_t chunk_tokens,
                  const int32_t *kspecs, int32_t nk, const int32_t *vspecs, int32_t nv,
                  const float *amax, const int32_t *lengths, const uint16_t *cdf_wire,
                  int64_t cdf_entries, const uint8_t *bytes, int64_t stream_bytes, uint8_t *out,
                  int64_t cap)
{
    int64_t need = orc_container_size(L, T, nk + nv, cdf_entries, stream_bytes);
    if (cap < need)
        return ORC_ERR_CAPACITY;
    uint8_t *p = out;
    memcpy(p, "CGKV", 4);
    put_u32(p + 4, 1u);
    put_u32(p + 8, (uint32_t)L);
    put_u32(p + 12, (uint32_t)T);
    put_u32(p + 16, (uint32_t)H);
    put_u32(p + 20, (uint32_t)D);
    put_u32(p + 24, (uint32_t)chunk_tokens);
    put_u32(p + 28, (uint32_t)nk);
    put_u32(p + 32, (uint32_t)nv);
    put_u32(p + 36, (uint32_t)orc_groups(T, chunk_tokens, NULL, NULL));
    put_u32(p + 40, (uint32_t)((uint64_t)stream_bytes & 0xFFFFFFFFu));
    put_u32(p + 44, (uint32_t)((uint64_t)stream_bytes >> 32));
    p += 48;
    for (int32_t i = 0; i < 3 * nk; ++i, p += 4)
        put_u32(p, (uint32_t)kspecs[i]);
    for (int32_t i = 0; i < 3 * nv; ++i, p += 4)
        put_u32(p, (uint32_t)vspecs[i]);
    for (int64_t i = 0; i < (int64_t)2 * L * T; ++i, p += 4) {
        uint32_t u;
        memcpy(&u, &amax[i], 4);
        put_u32(p, u);
    }
    for (int64_t i = 0; i < (int64_t)2 * L * T; ++i, p += 4)
        put_u32(p, (uint32_t)lengths[i]);
    for (int64_t i = 0; i < cdf_entries; ++i, p += 2) {
        p[0] = (uint8_t)cdf_wire[i];
        p[1] = (uint8_t)(cdf_wire[i] >> 8);
    }
    memcpy(p, bytes, (size_t)stream_bytes);
    return ORC_OK;
}

/* Threads OpenMP would use (1 when built without it). */
int32_t orc_max_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Int8 baseline codec                                                  */
/* ------------------------------------------------------------------ */

/* The reproduction page ("CacheGen复现项目：面向大模型服务的高效KV缓存压缩与流式传输
 * 方案", §编解码器模块) quantises KV to 8-bit integers with scale factors and
 * names no formula. Reading taken: the same symmetric scaling as
 * [CG-LMCache §2] with MAX = 127 and no offset, one scale per row (K/V,
 * layer, token): a = max_c |x_c|, f = 127 / a (0 when a = 0),
 * q = round_half_even(fp32(x * f)) in [-127, 127]; and the inverse of
 * [CG-LMCache §5] without offset: y = bf16(fp32(fp32(q / 127) * a)). */
int orc_int8_quantize_row(const uint16_t *x, int32_t C, float *scale, int8_t *q)
{
    float a = 0.0f;
    for (int32_t c = 0; c < C; ++c) {
        float v = fabsf(bf16_to_float(x[c]));
        if (!isfinite(v))
            return ORC_ERR_NONFINITE;
        if (v > a)
            a = v;
    }
    float f = (a == 0.0f) ? 0.0f : 127.0f / a;
    if (!isfinite(f)) /* as in orc_quantize_row */
        return ORC_ERR_NONFINITE;
    for (int32_t c = 0; c < C; ++c) {
        float y = bf16_to_float(x[c]) * f;
        int32_t iq = (int32_t)rintf(y);
        if (iq < -127 || iq > 127)
            return ORC_ERR_INVALID_ARG; /* cannot happen for finite input */
        q[c] = (int8_t)iq;
    }
    *scale = a;
    return ORC_OK;
}

void orc_int8_dequant_row(const int8_t *q, int32_t C, float a, uint16_t *y)
{
    for (int32_t c = 0; c < C; ++c) {
        float t = (float)q[c] / 127.0f;
        t = t * a;
        y[c] = float_to_bf16_rne(t);
    }
}

/* Whole blob: rows of C channels, row r at kv + r*C; q [rows][C],
 * scales [rows]. */
int orc_int8_encode(const uint16_t *kv, int64_t rows, int32_t C, int8_t *q, float *scales,
                    int32_t nthreads)
{
    int st = ORC_OK;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long long r = 0; r < (long long)rows; ++r) {
        int s = orc_int8_quantize_row(kv + (size_t)r * C, C, &scales[r], q + (size_t)r * C);
        if (s != ORC_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
            st = s;
        }
    }
    return st;
}

void orc_int8_decode(const int8_t *q, const float *scales, int64_t rows, int32_t C, uint16_t *kv,
                     int32_t nthreads)
{
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long long r = 0; r < (long long)rows; ++r)
        orc_int8_dequant_row(q + (size_t)r * C, C, scales[r], kv + (size_t)r * C);
}
