/*
 * cachegen.h: C ABI of the GB300 CacheGen KV-cache codec.
 *
 * The codec compresses a bf16 KV cache kv[L][2][T][H][D] (layers, K/V,
 * tokens, heads, head size; C = H*D channels) into
 *   - one fp32 scale per (K/V, layer, token): a = max_c |x|,
 *   - one 16-bit integer CDF per (token group, K/V, layer, channel),
 *   - one arithmetic-coded bitstream per (K/V, layer, token),
 * and decodes it back to bf16. The operation follows
 *   "LMCache 中的 KV Cache 压缩：CacheGen 编解码原理、配置方式与源码解析"
 *   (0539edu.com/news/4720135), cited below as [CG-LMCache]:
 *   §1 QuantizationSpec (per-layer bin counts), §2 Quantization,
 *   §3 CDF estimation and normalisation, §4 arithmetic coding in batches
 *   of at most 256 tokens, §5 decoding (prefix sum of stream lengths) and
 *   dequantisation;
 * with the 32-bit low/high arithmetic coder of Witten, Neal and Cleary
 * ("Arithmetic coding for data compression", CACM 30(6), 1987).
 *
 * Exact definitions (all integer results are bit-exact across runs):
 *   bins_l     bin count of layer l (from the K or V spec list); N = bins,
 *              MAX = bins/2 - 1; symbols lie in [0, 2*MAX].
 *   quantise   a = max_c |x_c|; f = MAX / a (fp32, f = 0 when a = 0);
 *              q = round_half_even(fp32(fp32(x * f) + MAX))  [CG-LMCache §2]
 *   groups     the T tokens form objects of chunk_tokens tokens (the last
 *              may be shorter); each object is cut into groups of at most
 *              256 tokens                                    [CG-LMCache §4]
 *   CDF        per (group, K/V, layer, channel), over the group's n tokens:
 *              cdf[i] = floor(cum[i] * (65536 - N) / n) + i, i = 0..N,
 *              cum[i] = number of symbols < i                [CG-LMCache §3]
 *   streams    one per (K/V, layer, token), holding the C symbols in
 *              channel order, coded with the channel's CDF: for r =
 *              high - low + 1, high = low + floor(r*cdf[s+1]/2^16) - 1,
 *              low = low + floor(r*cdf[s]/2^16), then the usual halving with
 *              pending bits; terminated by one more pending bit and then 0
 *              if low < 2^30 else 1, followed by the pending bits; bits MSB
 *              first, last byte zero-padded
 *   order      streams (and their lengths) are ordered group, then K/V,
 *              then layer, then token within the group; the byte stream is
 *              their concatenation; the decoder finds each stream by the
 *              exclusive prefix sum of the lengths           [CG-LMCache §5]
 *   dequantise y = bf16_rne(fp32(fp32((q - MAX) / MAX) * a))  [CG-LMCache §5]
 *
 * Buffers, layouts, ownership:
 *   The caller allocates every device buffer (kv, outputs, workspace) and
 *   keeps ownership; the library allocates only the host-side plan. All
 *   device pointers are plain device addresses. Calls that take a
 *   cudaStream_t enqueue work on it and return without waiting unless the
 *   comment says otherwise.
 *     kv         bf16 [L][2][T][H*D], 16-byte aligned
 *     amax       fp32 [2][L][T] (the scale a of each K/V, layer, token)
 *     lengths    int32 [2*L*T] stream lengths in bytes, stream order
 *     cdf        uint16 [cdf_entries]: per group, K/V, layer, channel the
 *                N+1 entries cdf[0..N] (cdf[N] = 65536 is stored as 0),
 *                16-byte aligned
 *     bytestream uint8, the concatenated streams, 16-byte aligned
 *
 * Threads: a plan holds two side streams and two events with which
 * cg_encode and cg_decode fork work onto a second stream and join it back
 * (cg_encode's side stream has the device's greatest stream priority, so
 * its smaller bin-count classes, whose tiles take longer, are dispatched
 * before the largest class and before lower-priority work). Calls that
 * use the same plan must therefore come from one host thread at a time (use
 * one plan per thread); calls on different plans are independent. Device
 * work of two calls may overlap only if they use different workspaces.
 *
 * Errors: argument and configuration errors are returned synchronously.
 * Errors found on the device (capacity exceeded, non-finite input, a
 * corrupt container) set a status word in the workspace; read it with
 * cg_last_device_error after the stream's work. Kernels never trap and
 * never wait on other blocks.
 */
#ifndef CACHEGEN_H
#define CACHEGEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cg_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* Layer range [start_layer, end_layer) with one bin count [CG-LMCache §1].
 * Per K and per V the ranges must cover [0, num_layers) exactly once;
 * bins must be even and in [4, 64]. */
typedef struct cg_quant_spec {
    int32_t start_layer;
    int32_t end_layer;
    int32_t bins;
} cg_quant_spec;

/* Shape of the KV blob and the codec configuration. num_heads*head_size
 * (C) must be a positive multiple of 8; chunk_tokens > 0 is the object
 * size in tokens [CG-LMCache §4: chunk_size]. */
typedef struct cg_config {
    int32_t num_layers;
    int32_t num_tokens;
    int32_t num_heads;
    int32_t head_size;
    int32_t chunk_tokens;
    const cg_quant_spec *kspecs;
    int32_t n_kspecs;
    const cg_quant_spec *vspecs;
    int32_t n_vspecs;
} cg_config;

typedef enum cg_status {
    CG_OK = 0,
    CG_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size */
    CG_ERR_SPEC = 2,        /* spec ranges do not tile [0, L) or bad bins */
    CG_ERR_CAPACITY = 3,    /* an output buffer is too small */
    CG_ERR_NONFINITE = 4,   /* the input holds inf or NaN, or a row too
                               small for a finite scale factor */
    CG_ERR_CORRUPT = 5,     /* a container or its tables are inconsistent */
    CG_ERR_TIMEOUT = 6,     /* a bounded device wait gave up (the decoder's
                               wait for a CDF table's bulk copy) */
    CG_ERR_CUDA = 7,        /* a CUDA runtime call failed */
    CG_ERR_UNSUPPORTED = 8  /* the shape exceeds this build's limits */
} cg_status;

typedef struct cg_plan cg_plan;

/* Sizes derived from a plan. */
typedef struct cg_sizes {
    size_t workspace_bytes;   /* device scratch that cg_encode/cg_decode need */
    size_t max_stream_bytes;  /* a bytestream capacity that can never overflow */
    size_t cdf_entries;       /* uint16 entries of the cdf buffer */
    size_t num_streams;       /* int32 entries of lengths (= 2*L*T) */
    size_t num_scales;        /* fp32 entries of amax (= 2*L*T) */
    size_t raw_bytes;         /* bytes of the bf16 KV blob (= 2*L*T*C*2) */
    int32_t num_groups;       /* token groups of at most 256 tokens */
    int32_t num_tiles;        /* groups * 2 * L */
    int32_t encode_launches;  /* kernels one cg_encode enqueues */
    int32_t decode_launches;  /* kernels one cg_decode enqueues */
    int32_t num_objects;      /* objects of chunk_tokens tokens (cg_object_range) */
} cg_sizes;

/* Device buffers of one encoded blob (all caller-owned). */
typedef struct cg_encoded {
    uint8_t *bytestream;
    size_t bytestream_capacity;
    int32_t *lengths;
    uint16_t *cdf;
    float *amax;
} cg_encoded;

/* Validate a configuration and build a plan (host memory only).
 * Returns CG_ERR_INVALID_ARG for null pointers or non-positive sizes,
 * CG_ERR_SPEC for spec lists that do not tile the layers or bad bins,
 * CG_ERR_UNSUPPORTED when the shape exceeds the kernels' limits
 * (L <= 256; C <= 4096 and C*(max bins+1)*2 bytes of CDF table must fit
 * in shared memory). [CG-LMCache §1] */
cg_status cg_plan_create(const cg_config *cfg, cg_plan **plan_out);

/* Free a plan (NULL is ignored). */
void cg_plan_destroy(cg_plan *plan);

/* Fill *out with the buffer sizes of a plan. Host only. */
cg_status cg_plan_sizes(const cg_plan *plan, cg_sizes *out);

/* The configuration a plan was built from (for a plan from
 * cg_container_open: the shape, chunk_tokens and spec lists recorded in the
 * container, which from_bytes of [CG-LMCache §5] must recover). Host only.
 * out gets the five sizes and n_kspecs / n_vspecs; its kspecs / vspecs
 * point at the caller's arrays kspecs[kcap] and vspecs[vcap], which receive
 * the spec triples in the order they were given. If kcap < n_kspecs or
 * vcap < n_vspecs nothing is copied and CG_ERR_CAPACITY is returned (the
 * counts are still set, so a caller can size its arrays and call again);
 * a NULL array is allowed with a capacity of 0. */
cg_status cg_plan_config(const cg_plan *plan, cg_config *out, cg_quant_spec *kspecs,
                         int32_t kcap, cg_quant_spec *vspecs, int32_t vcap);

/* Encode kv (device, bf16 [L][2][T][H*D]) into out's device buffers
 * [CG-LMCache §2-§4]. workspace (device, >= workspace_bytes, 256-byte
 * aligned) is scratch; its first 256 bytes receive the device status and
 * the total stream length, read back with cg_last_device_error. A
 * bytestream_capacity below the encoded size sets CG_ERR_CAPACITY on the
 * device and leaves the bytestream incomplete (never written out of
 * bounds); max_stream_bytes never overflows. Asynchronous on stream. */
cg_status cg_encode(const cg_plan *plan, const void *kv, void *workspace, size_t workspace_bytes,
                    const cg_encoded *out, cg_stream_t stream);

/* Decode in (device buffers written by cg_encode or cg_deserialize, with
 * stream_bytes bytes of streams; bytestream_capacity must be at least
 * stream_bytes rounded up to 16; stream_bytes below the number of
 * streams is CG_ERR_CORRUPT) into kv_out (device, bf16
 * [L][2][T][H*D], 16-byte aligned) [CG-LMCache §5]. With kv_out 32-byte
 * aligned and H*D a multiple of 16 every row is written in whole 32-byte
 * sectors (faster); otherwise in 16-byte pieces, with the same result.
 * Invalid CDF rows or lengths that do not add up to stream_bytes set
 * CG_ERR_CORRUPT on the device; a bounded wait inside the decoder that
 * runs out sets CG_ERR_TIMEOUT. Decoding of a corrupt stream still ends
 * after C symbols per stream and never reads outside the buffers.
 * Asynchronous on stream. */
cg_status cg_decode(const cg_plan *plan, const cg_encoded *in, uint64_t stream_bytes,
                    void *workspace, size_t workspace_bytes, void *kv_out, cg_stream_t stream);

/* Wait for stream, then read the device status word and the total stream
 * bytes of the last cg_encode/cg_decode that used this workspace (or the
 * status block of cg_encode_noalloc or cg_int8_encode; plan may be NULL,
 * the block's layout does not depend on it). Either output may be NULL.
 * Returns CG_ERR_CUDA if the copy fails. */
cg_status cg_last_device_error(const cg_plan *plan, const void *workspace, cg_status *status,
                               uint64_t *stream_bytes, cg_stream_t stream);

/* Bytes of the flat container for stream_bytes bytes of streams. The
 * container (little-endian) is: "CGKV", u32 version 1, i32 L, T, H, D,
 * chunk_tokens, n_kspecs, n_vspecs, num_groups, u64 stream_bytes; the
 * specs (K then V) as i32 triples; amax f32[2LT]; lengths i32[2LT]; cdf
 * u16[cdf_entries]; the streams. It replaces the pickled object of
 * [CG-LMCache §4]. */
cg_status cg_container_size(const cg_plan *plan, uint64_t stream_bytes, size_t *bytes);

/* Write the container of an encoded blob into host memory (pinned memory
 * copies fastest): header on the host, sections copied device-to-host.
 * Waits for stream before returning. */
cg_status cg_serialize(const cg_plan *plan, const cg_encoded *enc, uint64_t stream_bytes,
                       void *host_out, size_t host_capacity, size_t *written, cg_stream_t stream);

/* Read a container header from host memory and build its plan.
 * *stream_bytes gets the stream length. CG_ERR_CORRUPT for a bad magic,
 * version or inconsistent sizes. */
cg_status cg_container_open(const void *host_in, size_t len, cg_plan **plan_out,
                            uint64_t *stream_bytes);

/* Copy a container's sections from host memory into device buffers for
 * cg_decode. The plan must come from cg_container_open on the same bytes.
 * Waits for stream before returning. */
cg_status cg_deserialize(const cg_plan *plan, const void *host_in, size_t len,
                         const cg_encoded *dev_out, cg_stream_t stream);

/* Objects. LMCache keeps a KV cache as objects of chunk_tokens tokens
 * [CG-LMCache §4: chunk_size] (the last may be shorter). One cg_encode
 * codes every object of a plan in the same launches; since token groups
 * never span two objects, an object's CDF blocks, lengths and streams are
 * exactly those of encoding its tokens alone. The calls below cut an
 * encoded blob into one container per object, and put the containers of
 * all objects back into device buffers for one cg_decode.
 *
 * cg_object_range: first token and token count of object (0 <= object <
 * num_objects of cg_plan_sizes). Host only; CG_ERR_INVALID_ARG for an
 * object out of range.
 *
 * cg_object_streams: after a cg_encode (or cg_decode) that used this
 * workspace, the byte offset and length of the object's streams within the
 * bytestream, read from the workspace. Waits for stream.
 *
 * cg_object_container_size: bytes of the object's container for
 * stream_bytes bytes of streams. Host only.
 *
 * cg_serialize_object: write the object's container into host memory. It is
 * the container format of cg_serialize for a plan with the same L, H, D,
 * chunk_tokens and specs and T = the object's token count; its sections are
 * the object's amax columns [2][L][n], lengths, CDF blocks and streams, so it
 * is byte-identical to encoding and serialising the object's tokens alone.
 * Waits for stream.
 *
 * cg_deserialize_objects: copy the containers of all num_objects objects,
 * in object order (hosts[i] holds lens[i] bytes), into device buffers laid
 * out as cg_encode writes them for the whole plan; *stream_bytes gets the
 * total stream length to pass to cg_decode. Every header is checked before
 * anything is copied: CG_ERR_CORRUPT if a container is not object i of this
 * plan (shape, specs, tokens, groups, length), CG_ERR_CAPACITY if the
 * streams do not fit, CG_ERR_INVALID_ARG if num_objects differs from the
 * plan's. Waits for stream. */
cg_status cg_object_range(const cg_plan *plan, int32_t object, int32_t *first_token,
                          int32_t *num_tokens);
cg_status cg_object_streams(const cg_plan *plan, const void *workspace, int32_t object,
                            uint64_t *offset, uint64_t *bytes, cg_stream_t stream);
cg_status cg_object_container_size(const cg_plan *plan, int32_t object, uint64_t stream_bytes,
                                   size_t *bytes);
cg_status cg_serialize_object(const cg_plan *plan, const cg_encoded *enc, const void *workspace,
                              int32_t object, void *host_out, size_t host_capacity,
                              size_t *written, cg_stream_t stream);
cg_status cg_deserialize_objects(const cg_plan *plan, int32_t num_objects,
                                 const void *const *hosts, const size_t *lens,
                                 const cg_encoded *dev_out, uint64_t *stream_bytes,
                                 cg_stream_t stream);

/* Bytes of the fixed scratch array that cg_encode_noalloc uses (64 MiB). */
#define CG_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* Encode like cg_encode, but without a workspace argument and without any
 * device allocation: for callers that cannot allocate device memory when
 * they encode, such as a serving engine that has already reserved nearly
 * all of the GPU for its KV cache pool, or a latency-critical path where
 * cudaMalloc/cudaFree (which may synchronise the device) is not allowed.
 * The pages describe no such call; it is an addition of this library.
 * The scratch is one array of CG_NOALLOC_SCRATCH_BYTES bytes inside the
 * library, which every GPU that loads the library keeps until the process
 * exits. A plan whose workspace_bytes exceed it is rejected with
 * CG_ERR_UNSUPPORTED before anything is enqueued. The caller still passes
 * kv and the output buffers (same rules as cg_encode) and status_out, a
 * device buffer of at least 16 bytes that receives the device status word
 * and the total stream bytes (read it with cg_last_device_error, passing
 * status_out as the workspace). Every call looks up the array's device
 * address in the current device's context (nothing is cached, so a device
 * reset leaves no stale address); the first call on each device also loads
 * the library's device code there, so make that first call before any
 * stream capture. All calls share the one array and it keeps the last
 * call's contents (each call clears what must start at zero): calls that
 * can overlap on the GPU, from any stream or thread, race on it, so
 * serialise them. status_out is not a workspace: the object calls
 * (cg_object_streams, cg_serialize_object) read tile offsets that only a
 * cg_encode workspace holds, so they must not be given status_out; encode
 * with cg_encode when per-object containers are needed. Asynchronous on
 * stream. */
cg_status cg_encode_noalloc(const cg_plan *plan, const void *kv, const cg_encoded *out,
                            void *status_out, cg_stream_t stream);

/* Int8 baseline codec, the comparison point for the ratio and throughput
 * of the codec above. "CacheGen复现项目：面向大模型服务的高效KV缓存压缩与流式传输
 * 方案" (§编解码器模块) quantises KV to 8-bit integers with scale factors
 * and gives no formula; this library reads it as the symmetric scaling of
 * [CG-LMCache §2] with MAX = 127 and no offset, one scale per row:
 *   a = max_c |x_c|; f = 127 / a (fp32, f = 0 when a = 0);
 *   q = round_half_even(fp32(x * f)) in [-127, 127]  (int8)
 *   y = bf16_rne(fp32(fp32(q / 127) * a))
 * A row is C = channels bf16 values; for a KV cache, rows are the
 * (layer, K/V, token) rows of kv[L][2][T][H*D] in memory order, so
 * rows = 2*L*T and channels = H*D.
 *
 * cg_int8_encode: kv (device, bf16 [rows][channels], 16-byte aligned) into
 * q_out (device, int8 [rows][channels], 8-byte aligned) and scales_out
 * (device, fp32 [rows], the a of each row). status_out (device, 16 bytes,
 * 16-byte aligned) is cleared by the call; a row holding inf/NaN, or one
 * so small (a below about 2^-121) that 127 / a overflows fp32, sets its
 * first word to CG_ERR_NONFINITE (that row's q are then meaningless); read
 * it with cg_last_device_error(NULL, status_out, ...). channels is a
 * multiple of 8 up to 4096 (CG_ERR_INVALID_ARG, CG_ERR_UNSUPPORTED above);
 * rows = 0 only clears the status. Asynchronous on stream.
 *
 * cg_int8_decode: q and scales (device, as written by cg_int8_encode) into
 * kv_out (device, bf16 [rows][channels], 16-byte aligned). Every byte value
 * decodes (0x80, never written by the encoder, gives -128/127 * a).
 * Asynchronous on stream. */
cg_status cg_int8_encode(const void *kv, int64_t rows, int32_t channels, void *q_out,
                         float *scales_out, void *status_out, cg_stream_t stream);
cg_status cg_int8_decode(const void *q, const float *scales, int64_t rows, int32_t channels,
                         void *kv_out, cg_stream_t stream);

/* Per-kernel timing, for profiling. When enabled, each kernel that
 * cg_encode/cg_decode enqueue is bracketed by two CUDA events on the launch
 * stream (up to max_launches kernels are recorded; later ones are not).
 * cg_profile_read waits for the recorded events, reports per kernel name
 * the launches and the summed event time, and clears the record.
 * max_launches = 0 disables and frees the events. Not thread-safe: one
 * host thread per plan while profiling. */
typedef struct cg_kernel_profile {
    const char *kernel; /* static string */
    int64_t launches;
    double total_ms;
} cg_kernel_profile;

cg_status cg_profile_enable(cg_plan *plan, int32_t max_launches);
cg_status cg_profile_read(cg_plan *plan, cg_kernel_profile *out, int32_t capacity,
                          int32_t *count);

/* Human-readable name of a status code (static string). */
const char *cg_status_string(cg_status status);

#ifdef __cplusplus
}
#endif

#endif /* CACHEGEN_H */
