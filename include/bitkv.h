/*
 * bitkv.h -- C ABI of libbitkv.so: softmax attention over a 2-bit / mixed
 * FP16-INT4-INT2 / codebook quantised KV cache on NVIDIA B300 (sm_103a).
 *
 * Method sources (web pages on KV-cache quantisation for video generation):
 *   [JB]  "Quantized Keys Steal Attention: Bias Correction for KV-Cache
 *         Compression in Video Diffusion", abstract.
 *   [QWM] "QuantWM: Temporally Consistent 2-Bit KV Cache Quantization for
 *         Video World Models", Innovations and Methodology.
 *   [WQ]  WindowQuant paper note (zenn.dev), sections 何が新しいのか,
 *         技術的に面白い点, 実装者視点で気になった点.
 *
 * Conventions for every call:
 *   - Pointers marked (device) are CUDA device pointers owned by the caller;
 *     (host) pointers are ordinary host memory.  The library allocates no
 *     memory and keeps no state except a thread-local error message.
 *   - Tensors are row-major [B][H][L][d] with d contiguous, 16-byte aligned.
 *   - GQA: query head h reads kv head h / (Hq / Hkv).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device
 *     work is enqueued asynchronously; host-only calls are synchronous.
 *   - Every call returns a kv_status.  On failure nothing is launched (except
 *     KV_ERR_CUDA, reported after a failed launch) and kv_last_error() gives
 *     the reason.  Nothing throws across the ABI.
 */
#ifndef BITKV_H
#define BITKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,  /* bad size, null pointer, inconsistent arguments */
    KV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dtype/d/kind combination) */
    KV_ERR_CAPACITY = 3,     /* append would exceed the layout's block capacity */
    KV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than kv_attention_workspace() */
    KV_ERR_ALIGNMENT = 5,    /* a pointer is not 16-byte aligned */
    KV_ERR_CUDA = 6,         /* a CUDA launch or query failed */
    KV_ERR_TIMEOUT = 7,      /* a bounded device-side wait gave up: the output is incomplete.  Kernels run
                                asynchronously, so kv_attention reports it only through
                                kv_attention_status() (kv_attention_noalloc_status()), or at once
                                when the environment variable BITKV_DEBUG_SYNC is set */
    KV_ERR_RANGE = 8         /* an operand of the tensor-core path lies outside the fp16 range
                                (|x| >= 65520); reported like KV_ERR_TIMEOUT */
} kv_status;

typedef enum { KV_F32 = 0, KV_F16 = 1, KV_BF16 = 2 } kv_dtype;

/* Cache kinds.
 *   UNIFORM2 / UNIFORM4: every block INT2 / INT4 ([JB] INT2 cache with step sizes).
 *   MIXED: per-window FP16 / INT4 / INT2 chosen by kv_window_plan ([WQ]).
 *   CODEBOOK2: 2-bit centroid indices per key channel + INT2 values, with
 *              optional PSAC coefficients ([QWM]). */
typedef enum { KV_UNIFORM2 = 0, KV_UNIFORM4 = 1, KV_MIXED = 2, KV_CODEBOOK2 = 3 } kv_kind;

/* Segments of a (batch, kv-head) stream, in memory order ([WQ] 技術的に面白い点:
 * windows of one bit-width are stored together).  UNIFORM4 uses only the INT4
 * segment, UNIFORM2 and CODEBOOK2 only the INT2 segment. */
enum { KV_SEG_RAW16 = 0, KV_SEG_INT4 = 1, KV_SEG_INT2 = 2, KV_NUM_SEG = 3 };

typedef enum {
    KV_REGION_DATA = 0,      /* packed blocks: B * Hkv * stream_bytes bytes */
    KV_REGION_BLK_LEN = 1,   /* int32 [B][cap_total]: valid tokens per block */
    KV_REGION_BLK_POS = 2,   /* int32 [B][cap_total]: logical position of a block's first token */
    KV_REGION_CENTROIDS = 3, /* float [B][Hkv][d][4]: CODEBOOK2 key centroids */
    KV_REGION_PSAC_U = 4,    /* float [B][Hkv][d][r]: CODEBOOK2 PSAC basis (row-major d x r) */
    KV_REGION_RESID_VAR = 5  /* float [B][Hkv][d]: CODEBOOK2 per-channel key residual variances */
} kv_region;

/* Packed block format (32 token slots of one batch row and kv head).
 *   INT2/INT4 (b bits): Kc uint32[32][d*b/32] key codes token-major (channel c
 *     of token t at word t*(d*b/32) + c/(32/b), bit b*(c mod 32/b));
 *     Km float2[d] per-channel (step s, zero z); Vc uint32[d][b] value codes
 *     channel-major (token t of channel c at word c*b + t/(32/b), bit
 *     b*(t mod 32/b)); Vm float2[d/32][32] per-(32-channel group, token) (s, z).
 *   RAW16: K 16-bit[32][d] then V 16-bit[32][d] in raw_dtype; within each row
 *     the 16-byte chunk j of token t is stored at chunk position j XOR (t mod m),
 *     m = min(8, d/8) (so staged rows read conflict-free from shared memory).
 *   CODEBOOK2: Kc uint32[32][d/16] centroid indices token-major; Vc uint32[d][2];
 *     Vm float2[d/32][32]; Kq fp16[32][ceil8(r)] PSAC coefficients.
 * Quantisation ([JB] step sizes; [WQ] INT2/INT4): per group m = min, M = max,
 * s = fl32(fl32(M-m)/(2^b-1)), code = clamp(rint(fl32(fl32(x-m)/s)), 0, 2^b-1),
 * z = m; dequantised x = fmaf(code, s, z).  Key groups are 32 tokens of one
 * channel (one block, aligned to each appended chunk); value groups are 32
 * channels of one token.  Pad slots hold code 0 and zero metadata.
 * fp16 metadata (meta_dtype KV_F16; the smaller caches of [WQ] 主な結果 and the
 * QuantWM card's Key Results): Km is half2[d] and Vm half2[d/32][32], each pair
 * (s, z) as fp16 (d = 128 INT2: 3072 B per block instead of 4096).  s and z are
 * the fp16 round-to-nearest-even of the fp32 step and minimum (a -0 zero point
 * stored as +0), and the codes are taken against them:
 * code = clamp(rint(fl32(fl32(x-z16)/s16))), code 0 where s16 == 0.  The cached
 * values must lie within the fp16 range (|x| <= 65504). */
typedef struct {
    int32_t B, Hkv, d;          /* d: multiple of 32, <= 256 */
    int32_t kind;               /* kv_kind */
    int32_t raw_dtype;          /* MIXED: dtype of RAW16 blocks (KV_F16 or KV_BF16) */
    int32_t psac_rank;          /* CODEBOOK2: r in [0, 32] */
    int32_t cap_blocks[KV_NUM_SEG]; /* capacity per segment, in 32-token blocks */
    int32_t meta_dtype;         /* KV_F32 or KV_F16: dtype of the INT blocks' (s, z) metadata */
    /* derived by kv_layout_init: */
    int64_t block_bytes[KV_NUM_SEG];
    int64_t seg_offset[KV_NUM_SEG];
    int64_t stream_bytes;       /* bytes per (batch, kv head) */
} kv_layout;

/* A cache: the caller allocates every region (sizes from kv_layout_bytes),
 * zero-fills DATA, and keeps this struct on the host.  n_blocks / n_tokens
 * are host-side counters updated by kv_quantize_append.  resid_var is optional
 * and set by the caller after kv_cache_init: a CODEBOOK2 cache whose resid_var
 * holds the keys' residual variances (kv_codebook_residual_var) applies the
 * Jensen term to its codebook keys; with NULL they carry none. */
typedef struct {
    kv_layout layout;
    void* data;          /* (device) */
    int32_t* blk_len;    /* (device) */
    int32_t* blk_pos;    /* (device) */
    float* centroids;    /* (device) CODEBOOK2 only, else NULL */
    float* psac_u;       /* (device) CODEBOOK2 with psac_rank > 0, else NULL */
    int32_t n_blocks[KV_NUM_SEG];
    int32_t n_tokens;
    float* resid_var;    /* (device, nullable) CODEBOOK2: [B][Hkv][d] residual variances */
} kv_cache;

typedef struct {
    /* MIXED only: bit-width (16, 4 or 2) of each 32-token window of this
     * append, [B][ceil(n_tokens/32)], once in host memory (used for counts and
     * validation) and once on the device (read by the kernel). */
    const int8_t* window_bits_host;
    const int8_t* window_bits_dev;
} kv_append_opts;

typedef enum { KV_JENSEN_OFF = 0, KV_JENSEN_TAYLOR2 = 1, KV_JENSEN_EXACT = 2, KV_JENSEN_ISOTROPIC = 3 } kv_jensen;

typedef enum {
    KV_PATH_AUTO = 0,   /* decode kernel for n_q == 1, tensor-core kernel for bf16 d=128 chunks, else SIMT */
    KV_PATH_SIMT = 1,   /* CUDA-core fp32 kernel, any dtype/kind */
    KV_PATH_TC = 2,     /* tcgen05/TMEM kernel: bf16, d = 128, UNIFORM2 / UNIFORM4 / CODEBOOK2; CTA pairs
                           (2-CTA clusters, M = 256: each CTA expands half of every key and value tile) */
    KV_PATH_DECODE = 3, /* split-K streaming decode: n_q == 1, f16/bf16, d = 64 or 128 */
    KV_PATH_TC_SINGLE = 4 /* the tensor-core kernel with one CTA per query tile (M = 128) */
} kv_path;

typedef struct {
    float scale;         /* logit scale tau; 0 -> 1/sqrt(d) */
    int32_t jensen;      /* kv_jensen; applies to quantised cached keys only ([JB]) */
    int32_t psac;        /* 1: add tau (U^T q) . coeff for CODEBOOK2 caches ([QWM] PSAC) */
    int32_t out_f32;     /* 1: `out` is fp32 whatever the I/O dtype */
    int32_t num_splits;  /* key-range splits per (batch, head); 0 = automatic (the decode path
                            then launches one wave of resident CTAs, and streams past the first
                            (CTAs mod B Hkv) take one split fewer than kv_attention_plan reports) */
    int32_t path;        /* kv_path */
} kv_attn_opts;

typedef struct {
    double frac_fp16;    /* share of ranked windows kept FP16 (default 0.2) */
    double frac_int4;    /* share of ranked windows at INT4 (default 0.3) */
    int32_t force_first; /* 1: window 0 is FP16 regardless of similarity */
} kv_thresholds;

/* Fill a layout and its derived sizes.  Host only.  meta_dtype: KV_F32, or KV_F16 for
 * fp16 (s, z) metadata in the INT2 / INT4 blocks of UNIFORM2 / UNIFORM4 / MIXED caches
 * (KV_ERR_UNSUPPORTED for CODEBOOK2; KV_ERR_INVALID_ARG for another dtype). */
kv_status kv_layout_init(kv_layout* out, int B, int Hkv, int d, kv_kind kind, kv_dtype raw_dtype,
                         const int32_t cap_blocks[KV_NUM_SEG], int psac_rank, kv_dtype meta_dtype);

/* Bytes the caller must allocate for `region` (0 if the region is unused). */
size_t kv_layout_bytes(const kv_layout* layout, kv_region region);

/* Bind caller-allocated regions to a cache and zero its counters.  Host only;
 * checks null pointers and 16-byte alignment of `data`. */
kv_status kv_cache_init(kv_cache* cache, const kv_layout* layout, void* data, int32_t* blk_len,
                        int32_t* blk_pos, float* centroids, float* psac_u);

/* Quantise, pack and append one finished chunk ([JB]: the cache of previously
 * generated chunks; [WQ]: grouped layout).  K, V (device): [B][Hkv][n_tokens][d]
 * in `dtype`.  UNIFORM*: the chunk starts new blocks (the last may be partial).
 * MIXED: the cache position must be a multiple of 32, each window goes to the
 * segment of its bit-width; per-segment window counts must agree across B.
 * CODEBOOK2: centroids (and psac_u if r > 0) must be filled first.  With fp16
 * metadata the values must lie within the fp16 range.  Fails with
 * KV_ERR_CAPACITY before launching if a segment would overflow.  Updates
 * cache->n_blocks and cache->n_tokens on the host. */
kv_status kv_quantize_append(const void* K, const void* V, kv_dtype dtype, int n_tokens, kv_cache* cache,
                             const kv_append_opts* opts, void* stream);

/* Workspace bytes kv_attention needs for the same arguments (split partials). */
size_t kv_attention_workspace(const kv_cache* cache, kv_dtype dtype, int n_q, int n_cur, int Hq,
                              const kv_attn_opts* opts);

/* The kernel path (kv_path) and number of key-range splits kv_attention would
 * use for these arguments (on the decode path with automatic splits, the largest
 * count of any (batch, kv head)).  Host only; launches nothing.  One attention
 * call launches one kernel, plus one merge kernel when *splits_out > 1 on the
 * tensor-core and CUDA-core paths; the decode path always launches its kernel and
 * a merge kernel (which also writes the status words). */
kv_status kv_attention_plan(const kv_cache* cache, kv_dtype dtype, int n_q, int n_cur, int Hq,
                            const kv_attn_opts* opts, int32_t* path_out, int32_t* splits_out);

/* o_i = sum_j softmax_j(l_ij) v_j over the cache's valid tokens and the
 * current chunk ([JB]: chunk-wise autoregressive attention, current chunk
 * unquantised and bidirectional).  l_ij = tau q_i.k_hat_j - delta_ij (+ PSAC)
 * for cached keys, tau q_i.k_j for current keys.  Jensen delta ([JB]):
 * TAYLOR2 (tau^2/24) sum_c q_c^2 s_c^2, EXACT sum_c log(sinh x_c / x_c) with
 * x_c = tau q_c s_c / 2, ISOTROPIC (tau^2/24) |q|^2 mean_c s_c^2 (the query-norm
 * form; equal to TAYLOR2 when a group's steps are equal), using the step sizes
 * of the key's group; zero for RAW16 windows.  Codebook keys have no step size:
 * with cache->resid_var set, the second-order term of their residuals applies,
 * TAYLOR2 (tau^2/2) sum_c q'_c^2 v_c, ISOTROPIC (tau^2/2) |q'|^2 mean_c v_c, with
 * q' = q - U (U^T q) when opts->psac is on (PSAC restores the error along U) and
 * q' = q otherwise, one value per query row ([QWM] PSAC; [JB] second-order
 * correction); EXACT is KV_ERR_UNSUPPORTED there; without resid_var, none.
 * Precision: the result is defined over the exact dequantised entries
 * fmaf(code, s, z) (fp16 metadata: the fp16 entries fp16(code s + z)) and the
 * inputs as given.  The CUDA-core path (KV_PATH_SIMT) computes that definition in
 * fp32.  The decode path multiplies exact integer codes by the query scaled by
 * the step, split into fp16 high and low parts (about 22 bits), and adds the
 * zero-point term in fp32; with fp16 metadata it multiplies the fp16 entries by
 * the query taken as fp16 (a bf16 query beyond the fp16 range raises the range
 * flag).  The tensor-core path
 * holds the operands of both products in fp16: K_hat and V_hat are the fp16
 * roundings of the dequantised entries, Q and the current keys the fp16
 * conversions of their bf16 values (exact inside the fp16 range), P the fp16
 * rounding of the softmax weights; inputs or cache entries whose fp16 rounding
 * is infinite raise the range flag (KV_ERR_RANGE).  All paths accumulate in
 * fp32.  The 16-bit output is the round-to-nearest-even of the fp32 result.
 *   Q (device) [B][Hq][n_q][d]; Kcur, Vcur (device) [B][Hkv][n_cur][d] (may be
 *   NULL when n_cur == 0); out (device) [B][Hq][n_q][d] in dtype (fp32 if
 *   opts->out_f32); lse (device, nullable) fp32 [B][Hq][n_q] natural-log
 *   partition function.  workspace (device, 16-byte aligned) of ws_bytes >=
 *   kv_attention_workspace() (at least 256 bytes); it needs no initialisation.
 *   Its first 256 bytes are the call's status words: cleared by each call before
 *   its kernels run (tensor-core and CUDA-core paths) or written by the call's
 *   last kernel (decode path, from every CTA's own status word); read them with
 *   kv_attention_status() after the call.  Without BITKV_DEBUG_SYNC a
 *   KV_OK return means the work was queued, not that no device-side wait gave
 *   up. */
kv_status kv_attention(const void* Q, const void* Kcur, const void* Vcur, kv_dtype dtype, int n_q, int n_cur,
                       int Hq, const kv_cache* cache, const kv_attn_opts* opts, void* out, float* lse,
                       void* workspace, size_t ws_bytes, void* stream);

/* Status of the last kv_attention call that used `workspace` (device): waits for
 * the work queued on `stream`, copies the status words to the host and returns
 * KV_OK, KV_ERR_TIMEOUT (a bounded device-side wait gave up: that call's output
 * is incomplete) or KV_ERR_RANGE (see kv_attention).  Synchronous. */
kv_status kv_attention_status(const void* workspace, void* stream);

/* kv_attention without a workspace argument, for callers that cannot allocate
 * device memory: code running where cudaMalloc is unavailable or not allowed
 * (a host callback, an allocator hook, a plug-in given only its input and
 * output buffers, a process whose device memory belongs to another
 * framework).  The source pages have no counterpart; this is a library
 * convenience.
 *   Arguments, layouts, results and errors are those of kv_attention.  The
 *   scratch kv_attention would take from `workspace` comes from one fixed
 *   device array of KV_NOALLOC_SCRATCH_BYTES inside the library, which every
 *   GPU that loads the library holds until the process exits.  The call
 *   allocates and frees nothing.
 *   With opts->num_splits == 0 the key range is split as kv_attention would
 *   split it, or less where the partials would not fit; sizes whose scratch
 *   still exceeds the array (or an explicit num_splits that does) are rejected
 *   with KV_ERR_WORKSPACE before anything is launched.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  All calls share the one array and find the previous call's
 *   contents in it (the kernels clear what must start at zero), so calls that
 *   overlap on the GPU -- on different streams, or from several host threads
 *   -- race and give wrong results: serialise them. */
#define KV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
kv_status kv_attention_noalloc(const void* Q, const void* Kcur, const void* Vcur, kv_dtype dtype, int n_q,
                               int n_cur, int Hq, const kv_cache* cache, const kv_attn_opts* opts, void* out,
                               float* lse, void* stream);

/* kv_attention_status() for the last kv_attention_noalloc call on the current
 * device: reads the status words in the library's fixed array after the work
 * queued on `stream`.  Synchronous.  The array's device address is looked up once
 * per device and kept; after cudaDeviceReset() (or any re-creation of the
 * device's primary context) the kept address is stale, so neither no-alloc call
 * may be used again in that process. */
kv_status kv_attention_noalloc_status(void* stream);

/* Per-window bit-widths from window/question similarity ([WQ] 何が新しいのか
 * table, 技術的に面白い点: first window FP16).  Host only.  sim (host) [n_windows];
 * windows 1..W-1 (0..W-1 if !force_first) ranked by sim descending, ties to
 * the lower index; ranks [0, floor(f16*n)) FP16, [.., floor((f16+f4)*n)) INT4,
 * the rest INT2 (fp64 arithmetic).  bits_out (host) [n_windows] in {16,4,2};
 * perm_out (host, nullable) [n_windows]: window stored at each physical block
 * (FP16, then INT4, then INT2, ascending window index within each). */
kv_status kv_window_plan(const float* sim, int n_windows, const kv_thresholds* th, int8_t* bits_out,
                         int32_t* perm_out);

/* The similarity kv_window_plan ranks by ([WQ] 何が新しいのか: each window's
 * cosine similarity to the text question): for every 32-token window w of K,
 * cos(u_w, v) with u_w the mean of the window's valid tokens' keys and v the
 * mean of the question tokens' keys, all Hkv heads' d channels concatenated;
 * 0 where either is the zero vector (or m == 0).  fp32 sums on the device.
 *   K (device) [B][Hkv][n][d], Kq (device) [B][Hkv][m][d], both in dtype and
 *   16-byte aligned, d * sizeof(dtype) a multiple of 16 and Hkv * d at most
 *   1024 16-byte groups and B at most 65535 (KV_ERR_UNSUPPORTED otherwise);
 *   sim (device, fp32) [B][ceil(n / 32)], written by the call (copy it to the
 *   host for kv_window_plan).  n == 0 does nothing.  Async on `stream`. */
kv_status kv_window_similarity(const void* K, const void* Kq, kv_dtype dtype, int B, int Hkv, int n, int m, int d,
                               float* sim, void* stream);

/* Fit CODEBOOK2 key centroids ([QWM] QSAC): per (b, kv head, channel) 1-D
 * Lloyd k-means, 4 centroids, quantile init x_(floor((2k+1)n/8)) of the sorted
 * values, `iters` iterations, nearest by fp64 |x - mu| (ties to the lower index),
 * fp64 member sums (exact for 16-bit inputs at these sizes), empty clusters
 * keep their centroid.  K (device) [B][Hkv][n_tokens][d] (bf16/f16/f32),
 * n_tokens <= 32768; writes cache->centroids as fp32 [B][Hkv][d][4].
 * Qhist (device, nullable) [B][Hkv][n_hist][d] in dtype: if given, the
 * per-channel sensitivity mean q_c^2 is written to weights_out (device,
 * [B][Hkv][d] fp32); it is a per-channel constant and does not change the
 * centroids.  Needs no workspace (kv_codebook_workspace() returns 0). */
size_t kv_codebook_workspace(const kv_layout* layout, int n_tokens);
kv_status kv_codebook_fit(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, int iters,
                          const void* Qhist, int n_hist, float* weights_out, void* workspace, size_t ws_bytes,
                          void* stream);

/* PSAC basis ([QWM] principal-subspace compensation): for each (b, kv head) the
 * top-r eigenvectors of the uncentred second moment (1/n) sum q q^T of the
 * historical queries Qhist (device) [B][Hkv][n_hist][d], eigenvalues
 * descending (ties to the lower index), the largest-magnitude entry of each
 * made positive.  Writes cache->psac_u (fp32 [d][r]) and, if eigvals_out
 * (device) is non-null, the r eigenvalues [B][Hkv][r].  The second moment is
 * accumulated in fp64 and diagonalised by a cyclic Jacobi method in fp64 on
 * the device (d even, <= 128); workspace (device) >= kv_psac_workspace() =
 * 2 B Hkv d^2 doubles. */
/* QSAC with residual ranges ([QWM] QSAC: the clustering weighs the historical
 * queries' sensitivity together with the range of the residuals, protecting the
 * channels that matter more).  As kv_codebook_fit, with Qhist and weights_out
 * required: the weights w_c are computed first, channel c gets the relative
 * sensitivity rho_c = w_c / max_c' w_c' of its (b, kv head) (fp64 of the fp32
 * weights; 0 when all are 0), and every update moves a cluster's member mean
 * towards its mid-range (min + max) / 2, mu_k = mean_k + rho_c (mid_k - mean_k), each
 * fp64 operation rounded once in that order: rho = 0 is Lloyd, the most sensitive
 * channel minimises its largest residual.  Centroids fp32 as kv_codebook_fit. */
kv_status kv_codebook_fit_range(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, int iters,
                                const void* Qhist, int n_hist, float* weights_out, void* stream);

/* Residual variances of codebook keys, for the Jensen term of CODEBOOK2 caches:
 * v_c = (1/n) sum_t (k_tc - mu_a)^2 over K (device) [B][Hkv][n_tokens][d] in dtype
 * against the cache's fp32 centroids, a = the nearest centroid (fp64 distance,
 * ties to the lower index, the index the append stores), summed in fp64 and
 * stored as fp32 in cache->resid_var (which must be set).  Async on `stream`. */
kv_status kv_codebook_residual_var(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, void* stream);

size_t kv_psac_workspace(const kv_layout* layout);
kv_status kv_psac_basis(const void* Qhist, kv_dtype dtype, int n_hist, kv_cache* cache, float* eigvals_out,
                        void* workspace, size_t ws_bytes, void* stream);

/* Debug: write the cache's dequantised entries fmaf(code, s, z) (codebook keys:
 * the centroid; RAW16 entries as stored) as fp32 in logical token order, K_out
 * and V_out (device) [B][Hkv][n_tokens][d].  Computed by the device routine the
 * CUDA-core attention kernel (KV_PATH_SIMT) reads the cache with; the tensor-core
 * and decode kernels expand the cache with their own routines, which
 * kv_debug_operands() exposes.  Positions never appended are left untouched. */
kv_status kv_dequantize(const kv_cache* cache, float* K_out, float* V_out, void* stream);

/* Debug: the cache operands an attention kernel builds for its products, made by
 * that kernel's own device routines and written in stream slot order: K_out and
 * V_out (device, 16-byte aligned) fp16 [B][Hkv][32 n][d], n the cache's blocks
 * over all segments in memory order (FP16, INT4, INT2), token t of block i at
 * slot 32 i + t (pad slots included).
 *   path KV_PATH_TC (UNIFORM2 / UNIFORM4 / CODEBOOK2, d 128): the tensor-core
 *     kernel's K_hat and V_hat (the fp16 roundings of the dequantised entries; with
 *     fp16 metadata the entries themselves, which are fp16 numbers), expanded by its
 *     producer routines from a staged tile and un-swizzled.
 *   path KV_PATH_DECODE (UNIFORM2 / UNIFORM4 / MIXED, d 64 or 128): with fp32
 *     metadata the decode kernel forms no dequantised entry: its key and value
 *     operands are the codes, as the exact fp16 integers its extraction routine
 *     feeds the MMAs; with fp16 metadata they are the fp16 entries.  FP16 slots are
 *     not written (that path reads them as stored).
 * Async on `stream`. */
kv_status kv_debug_operands(const kv_cache* cache, int path, void* K_out, void* V_out, void* stream);

/* Message of the last failure on this thread ("" if none). */
const char* kv_last_error(void);

/* Library version string. */
const char* kv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BITKV_H */
