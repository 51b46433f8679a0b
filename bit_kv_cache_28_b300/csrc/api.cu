// C ABI entry points of libbitkv: argument checks, layout arithmetic, the
// host-side window plan, and dispatch to the kernels.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <numeric>
#include <string>
#include <vector>

#include "common.cuh"

namespace bitkv {

// kernels (other translation units)
kv_status launch_append(const void* K, const void* V, kv_dtype dt, int n_tokens, const kv_cache* cache, int mode,
                        int uni_seg, const int8_t* win_bits, int n_win, int grid_x, cudaStream_t st);
kv_status launch_dequant(const kv_cache* cache, float* Kout, float* Vout, cudaStream_t st);
kv_status launch_tc_operands(const kv_cache* cache, void* Kout, void* Vout, cudaStream_t st);
kv_status launch_dec_operands(const kv_cache* cache, void* Kout, void* Vout, cudaStream_t st);
kv_status launch_attn_simt(const void* Q, const void* Kc, const void* Vc, kv_dtype dt, int n_q, int n_cur, int Hq,
                           const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out,
                           int out_f32, float* lse, void* ws, cudaStream_t st);
size_t simt_workspace(const kv_cache* cache, int n_q, int Hq, int n_splits);
int simt_units_cache(const kv_cache* c);
kv_status launch_attn_decode(const void* Q, const void* Kc, const void* Vc, kv_dtype dt, int n_cur, int Hq,
                             const kv_cache* cache, float tau, int jensen, int n_splits, int n_ctas, void* out, int out_f32,
                             float* lse, void* ws, cudaStream_t st);
size_t decode_workspace(const kv_cache* cache, int Hq, int n_splits);
int decode_auto_splits(const kv_cache* cache, int Hq);
int decode_auto_ctas(const kv_cache* cache, int Hq, int n_splits);
bool decode_supported(const kv_cache* cache, kv_dtype dt, int n_q, int Hq);
kv_status launch_attn_tc(const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                         const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out, int out_f32,
                         float* lse, void* ws, bool pair, cudaStream_t st);
size_t tc_workspace(const kv_cache* cache, int n_q, int Hq, int n_splits);
int tc_auto_splits(const kv_cache* cache, int n_q, int n_cur, int Hq, bool pair);
bool tc_supported(const kv_cache* cache, kv_dtype dt, int n_q, int Hq, const char** why);
kv_status launch_codebook_fit(const void* K, kv_dtype dt, int n_tokens, const kv_cache* cache, int iters,
                              const void* Qhist, int n_hist, float* weights_out, int range, void* ws, cudaStream_t st);
kv_status launch_residual_var(const void* K, kv_dtype dt, int n_tokens, const kv_cache* cache, cudaStream_t st);
size_t codebook_ws_bytes(const kv_layout* L, int n_tokens);
kv_status launch_psac_basis(const void* Qhist, kv_dtype dt, int n_hist, const kv_cache* cache, float* eig_out,
                            void* ws, cudaStream_t st);
size_t psac_ws_bytes(const kv_layout* L);

static thread_local std::string g_err;

kv_status set_error(kv_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

kv_status check_launch(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    if (getenv("BITKV_DEBUG_SYNC")) {
        const cudaError_t e2 = cudaDeviceSynchronize();
        if (e2 != cudaSuccess) return set_error(KV_ERR_CUDA, "%s (sync): %s", what, cudaGetErrorString(e2));
    }
    return KV_OK;
}

kv_status clear_device(void* p, size_t bytes, cudaStream_t st, const char* who) {
    const cudaError_t e = cudaMemsetAsync(p, 0, bytes, st);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "%s: clearing %zu bytes of workspace: %s", who, bytes,
                                           cudaGetErrorString(e));
    return KV_OK;
}

kv_status read_status(const void* ws, cudaStream_t st) {
    int h[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "reading the attention status: %s", cudaGetErrorString(e));
    if (h[0] != 0)
        return set_error(KV_ERR_TIMEOUT, "a bounded device-side wait gave up (wait %d); the output is incomplete", h[0]);
    if (h[1] != 0)
        return set_error(KV_ERR_RANGE, "an operand of the tensor-core path lies outside the fp16 range (|x| >= 65520)");
    return KV_OK;
}

kv_status set_smem_limit(const void* kernel, size_t bytes, const char* name) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> limits;   // (kernel, device) -> bytes set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "%s: cudaGetDevice: %s", name, cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = limits[{kernel, dev}];
    if (bytes <= have) return KV_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess)
        return set_error(KV_ERR_CUDA, "%s: %zu bytes of shared memory: %s", name, bytes, cudaGetErrorString(e));
    have = bytes;
    return KV_OK;
}

static int ceil8(int r) { return (r + 7) / 8 * 8; }

static long long block_bytes_of(int cls, int d, int r, int meta16) {
    const long long pair = meta16 ? 4 : 8;    // bytes of one (s, z)
    switch (cls) {
        case CLS_RAW16: return 2LL * kBlockTokens * d * 2;
        case CLS_INT4: return 2LL * (kBlockTokens * d * 4 / 8) + 2 * pair * d;
        case CLS_INT2: return 2LL * (kBlockTokens * d * 2 / 8) + 2 * pair * d;
        case CLS_CB2: return 2LL * (kBlockTokens * d * 2 / 8) + 8LL * d + kBlockTokens * ceil8(r) * 2LL;
    }
    return 0;
}

DevCache make_dev_cache(const kv_cache* cc) {
    const kv_layout& L = cc->layout;
    DevCache c;
    c.data = static_cast<unsigned char*>(cc->data);
    c.blk_len = cc->blk_len;
    c.blk_pos = cc->blk_pos;
    c.centroids = cc->centroids;
    c.psac_u = cc->psac_u;
    c.resid_var = cc->layout.kind == KV_CODEBOOK2 ? cc->resid_var : nullptr;
    c.B = L.B;
    c.Hkv = L.Hkv;
    c.d = L.d;
    c.kind = L.kind;
    c.raw_dtype = L.raw_dtype;
    c.r = L.psac_rank;
    c.rp = ceil8(L.psac_rank);
    c.meta16 = L.meta_dtype == KV_F16;
    c.cap_total = L.cap_blocks[0] + L.cap_blocks[1] + L.cap_blocks[2];
    int base = 0;
    for (int s = 0; s < KV_NUM_SEG; ++s) {
        c.seg_base[s] = base;
        base += L.cap_blocks[s];
        c.n_blocks[s] = cc->n_blocks[s];
        c.block_bytes[s] = L.block_bytes[s];
        c.seg_offset[s] = L.seg_offset[s];
    }
    c.stream_bytes = L.stream_bytes;
    return c;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int dtype_size(kv_dtype dt) { return dt == KV_F32 ? 4 : 2; }

static kv_status check_cache(const kv_cache* c) {
    if (!c) return set_error(KV_ERR_INVALID_ARG, "cache is NULL");
    const kv_layout& L = c->layout;
    if (L.B <= 0 || L.Hkv <= 0 || L.d <= 0) return set_error(KV_ERR_INVALID_ARG, "cache layout not initialised");
    if (!c->data || !c->blk_len || !c->blk_pos) return set_error(KV_ERR_INVALID_ARG, "cache regions not bound");
    for (int s = 0; s < KV_NUM_SEG; ++s)
        if (c->n_blocks[s] < 0 || c->n_blocks[s] > L.cap_blocks[s])
            return set_error(KV_ERR_INVALID_ARG, "cache counters out of range");
    return KV_OK;
}

}  // namespace bitkv

using namespace bitkv;

extern "C" {

const char* kv_last_error(void) { return g_err.c_str(); }

const char* kv_version(void) { return "bitkv 0.1 (sm_103a)"; }

kv_status kv_layout_init(kv_layout* out, int B, int Hkv, int d, kv_kind kind, kv_dtype raw_dtype,
                         const int32_t cap_blocks[KV_NUM_SEG], int psac_rank, kv_dtype meta_dtype) {
    if (!out || !cap_blocks) return set_error(KV_ERR_INVALID_ARG, "layout or cap_blocks is NULL");
    if (B <= 0 || Hkv <= 0) return set_error(KV_ERR_INVALID_ARG, "B=%d Hkv=%d must be positive", B, Hkv);
    if (d <= 0 || d % 32 != 0 || d > 256) return set_error(KV_ERR_UNSUPPORTED, "d=%d must be a multiple of 32 <= 256", d);
    if (kind < KV_UNIFORM2 || kind > KV_CODEBOOK2) return set_error(KV_ERR_INVALID_ARG, "unknown kind %d", (int)kind);
    if (psac_rank < 0 || psac_rank > 32) return set_error(KV_ERR_INVALID_ARG, "psac_rank=%d not in [0,32]", psac_rank);
    if (kind != KV_CODEBOOK2 && psac_rank != 0) return set_error(KV_ERR_INVALID_ARG, "psac_rank needs a CODEBOOK2 cache");
    if (kind == KV_MIXED && raw_dtype != KV_F16 && raw_dtype != KV_BF16)
        return set_error(KV_ERR_INVALID_ARG, "MIXED caches store 16-bit windows: raw_dtype must be F16 or BF16");
    if (meta_dtype != KV_F32 && meta_dtype != KV_F16)
        return set_error(KV_ERR_INVALID_ARG, "meta_dtype must be KV_F32 or KV_F16");
    if (meta_dtype == KV_F16 && kind == KV_CODEBOOK2)
        return set_error(KV_ERR_UNSUPPORTED, "fp16 metadata is for UNIFORM2 / UNIFORM4 / MIXED caches");
    for (int s = 0; s < KV_NUM_SEG; ++s)
        if (cap_blocks[s] < 0) return set_error(KV_ERR_INVALID_ARG, "negative capacity");
    const bool used[3] = {kind == KV_MIXED, kind == KV_MIXED || kind == KV_UNIFORM4,
                          kind == KV_MIXED || kind == KV_UNIFORM2 || kind == KV_CODEBOOK2};
    for (int s = 0; s < KV_NUM_SEG; ++s)
        if (!used[s] && cap_blocks[s] != 0)
            return set_error(KV_ERR_INVALID_ARG, "segment %d is unused by this kind and needs capacity 0", s);
    kv_layout L;
    memset(&L, 0, sizeof(L));
    L.B = B;
    L.Hkv = Hkv;
    L.d = d;
    L.kind = kind;
    L.raw_dtype = raw_dtype;
    L.psac_rank = psac_rank;
    L.meta_dtype = meta_dtype;
    long long off = 0;
    for (int s = 0; s < KV_NUM_SEG; ++s) {
        L.cap_blocks[s] = cap_blocks[s];
        L.block_bytes[s] = block_bytes_of(seg_class(kind, s), d, psac_rank, meta_dtype == KV_F16);
        L.seg_offset[s] = off;
        off += (long long)cap_blocks[s] * L.block_bytes[s];
    }
    L.stream_bytes = off;
    *out = L;
    return KV_OK;
}

size_t kv_layout_bytes(const kv_layout* L, kv_region region) {
    if (!L) return 0;
    const long long cap = (long long)L->cap_blocks[0] + L->cap_blocks[1] + L->cap_blocks[2];
    switch (region) {
        case KV_REGION_DATA: return (size_t)L->B * L->Hkv * L->stream_bytes;
        case KV_REGION_BLK_LEN:
        case KV_REGION_BLK_POS: return (size_t)L->B * cap * sizeof(int32_t);
        case KV_REGION_CENTROIDS:
            return L->kind == KV_CODEBOOK2 ? (size_t)L->B * L->Hkv * L->d * 4 * sizeof(float) : 0;
        case KV_REGION_PSAC_U:
            return L->kind == KV_CODEBOOK2 ? (size_t)L->B * L->Hkv * L->d * L->psac_rank * sizeof(float) : 0;
        case KV_REGION_RESID_VAR:
            return L->kind == KV_CODEBOOK2 ? (size_t)L->B * L->Hkv * L->d * sizeof(float) : 0;
    }
    return 0;
}

kv_status kv_cache_init(kv_cache* c, const kv_layout* L, void* data, int32_t* blk_len, int32_t* blk_pos,
                        float* centroids, float* psac_u) {
    if (!c || !L) return set_error(KV_ERR_INVALID_ARG, "cache or layout is NULL");
    if (!data || !blk_len || !blk_pos) return set_error(KV_ERR_INVALID_ARG, "data/blk_len/blk_pos must be set");
    if (!aligned16(data)) return set_error(KV_ERR_ALIGNMENT, "cache data must be 16-byte aligned");
    if (L->kind == KV_CODEBOOK2 && !centroids) return set_error(KV_ERR_INVALID_ARG, "CODEBOOK2 needs centroids");
    if (L->kind == KV_CODEBOOK2 && L->psac_rank > 0 && !psac_u)
        return set_error(KV_ERR_INVALID_ARG, "psac_rank > 0 needs psac_u");
    memset(c, 0, sizeof(*c));
    c->layout = *L;
    c->data = data;
    c->blk_len = blk_len;
    c->blk_pos = blk_pos;
    c->centroids = centroids;
    c->psac_u = psac_u;
    return KV_OK;
}

kv_status kv_quantize_append(const void* K, const void* V, kv_dtype dtype, int n_tokens, kv_cache* cache,
                             const kv_append_opts* opts, void* stream) {
    AbiRange nvtx_range("kv_quantize_append");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    const kv_layout& L = cache->layout;
    if (!K || !V) return set_error(KV_ERR_INVALID_ARG, "K or V is NULL");
    if (!aligned16(K) || !aligned16(V)) return set_error(KV_ERR_ALIGNMENT, "K and V must be 16-byte aligned");
    if (dtype < KV_F32 || dtype > KV_BF16) return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (n_tokens <= 0) return set_error(KV_ERR_INVALID_ARG, "n_tokens=%d must be positive", n_tokens);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nb = (n_tokens + kBlockTokens - 1) / kBlockTokens;
    if (L.kind == KV_UNIFORM2 || L.kind == KV_UNIFORM4) {
        const int seg = L.kind == KV_UNIFORM4 ? KV_SEG_INT4 : KV_SEG_INT2;
        if (cache->n_blocks[seg] + nb > L.cap_blocks[seg])
            return set_error(KV_ERR_CAPACITY, "append of %d blocks exceeds capacity (%d of %d used)", nb,
                             cache->n_blocks[seg], L.cap_blocks[seg]);
        s = launch_append(K, V, dtype, n_tokens, cache, 0, seg, nullptr, 0, nb, st);
        if (s != KV_OK) return s;
        cache->n_blocks[seg] += nb;
    } else if (L.kind == KV_MIXED) {
        if (!opts || !opts->window_bits_host || !opts->window_bits_dev)
            return set_error(KV_ERR_INVALID_ARG, "MIXED append needs window bits on host and device");
        if (cache->n_tokens % kBlockTokens != 0)
            return set_error(KV_ERR_INVALID_ARG, "MIXED append must start at a multiple of 32 tokens (at %d)",
                             cache->n_tokens);
        if ((int)dtype != L.raw_dtype)
            return set_error(KV_ERR_UNSUPPORTED, "MIXED append dtype must equal the layout's raw_dtype");
        int counts[3] = {0, 0, 0};
        for (int b = 0; b < L.B; ++b) {
            int cb[3] = {0, 0, 0};
            for (int w = 0; w < nb; ++w) {
                const int bits = opts->window_bits_host[(long long)b * nb + w];
                if (bits == 16) ++cb[0];
                else if (bits == 4) ++cb[1];
                else if (bits == 2) ++cb[2];
                else return set_error(KV_ERR_INVALID_ARG, "window bits must be 16, 4 or 2 (got %d)", bits);
            }
            if (b == 0) memcpy(counts, cb, sizeof(cb));
            else if (memcmp(counts, cb, sizeof(cb)) != 0)
                return set_error(KV_ERR_INVALID_ARG, "per-segment window counts differ across the batch");
        }
        for (int sg = 0; sg < KV_NUM_SEG; ++sg)
            if (cache->n_blocks[sg] + counts[sg] > L.cap_blocks[sg])
                return set_error(KV_ERR_CAPACITY, "segment %d: %d + %d blocks exceed capacity %d", sg,
                                 cache->n_blocks[sg], counts[sg], L.cap_blocks[sg]);
        s = launch_append(K, V, dtype, n_tokens, cache, 1, 0, opts->window_bits_dev, nb, nb, st);
        if (s != KV_OK) return s;
        for (int sg = 0; sg < KV_NUM_SEG; ++sg) cache->n_blocks[sg] += counts[sg];
    } else {
        if (!cache->centroids) return set_error(KV_ERR_INVALID_ARG, "CODEBOOK2 append needs fitted centroids");
        if (L.psac_rank > 0 && !cache->psac_u) return set_error(KV_ERR_INVALID_ARG, "PSAC basis not bound");
        const int seg = KV_SEG_INT2;
        if (cache->n_blocks[seg] + nb > L.cap_blocks[seg])
            return set_error(KV_ERR_CAPACITY, "append of %d blocks exceeds capacity", nb);
        s = launch_append(K, V, dtype, n_tokens, cache, 2, seg, nullptr, 0, nb, st);
        if (s != KV_OK) return s;
        cache->n_blocks[seg] += nb;
    }
    cache->n_tokens += n_tokens;
    return KV_OK;
}

static int pick_path(const kv_cache* cache, kv_dtype dt, int n_q, int Hq, const kv_attn_opts* o) {
    if (o && o->path != KV_PATH_AUTO) return o->path;
    if (decode_supported(cache, dt, n_q, Hq)) return KV_PATH_DECODE;
    const char* why = nullptr;
    if (tc_supported(cache, dt, n_q, Hq, &why)) return KV_PATH_TC;
    return KV_PATH_SIMT;
}

static int pick_splits(const kv_cache* cache, int path, int n_q, int n_cur, int Hq, const kv_attn_opts* o) {
    if (o && o->num_splits > 0) return o->num_splits;
    if (path == KV_PATH_DECODE) return decode_auto_splits(cache, Hq);
    if (path == KV_PATH_TC || path == KV_PATH_TC_SINGLE)
        return tc_auto_splits(cache, n_q, n_cur, Hq, path == KV_PATH_TC);
    // SIMT: enough CTAs to fill the GPU about twice
    const long long ctas = (long long)cache->layout.B * Hq * ((n_q + 31) / 32);
    const int units = simt_units_cache(cache) + (n_cur + 31) / 32;
    int sp = (int)std::max<long long>(1, (2 * 148 + ctas - 1) / std::max<long long>(ctas, 1));
    return std::max(1, std::min(sp, std::max(units, 1)));
}

size_t kv_attention_workspace(const kv_cache* cache, kv_dtype dt, int n_q, int n_cur, int Hq,
                              const kv_attn_opts* opts) {
    if (!cache || n_q <= 0 || Hq <= 0) return 0;
    const int path = pick_path(cache, dt, n_q, Hq, opts);
    const int sp = pick_splits(cache, path, n_q, n_cur, Hq, opts);
    if (path == KV_PATH_DECODE) return decode_workspace(cache, Hq, sp);
    if (path == KV_PATH_TC || path == KV_PATH_TC_SINGLE) return tc_workspace(cache, n_q, Hq, sp);
    return simt_workspace(cache, n_q, Hq, sp);
}

kv_status kv_attention_plan(const kv_cache* cache, kv_dtype dtype, int n_q, int n_cur, int Hq,
                            const kv_attn_opts* opts, int32_t* path_out, int32_t* splits_out) {
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (n_q <= 0 || n_cur < 0 || Hq <= 0) return set_error(KV_ERR_INVALID_ARG, "bad sizes");
    const int path = pick_path(cache, dtype, n_q, Hq, opts);
    if (path_out) *path_out = path;
    if (splits_out) *splits_out = pick_splits(cache, path, n_q, n_cur, Hq, opts);
    return KV_OK;
}

kv_status kv_attention(const void* Q, const void* Kcur, const void* Vcur, kv_dtype dtype, int n_q, int n_cur, int Hq,
                       const kv_cache* cache, const kv_attn_opts* opts, void* out, float* lse, void* workspace,
                       size_t ws_bytes, void* stream) {
    AbiRange nvtx_range("kv_attention");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    const kv_layout& L = cache->layout;
    if (!Q || !out) return set_error(KV_ERR_INVALID_ARG, "Q or out is NULL");
    if (n_q <= 0 || n_cur < 0 || Hq <= 0) return set_error(KV_ERR_INVALID_ARG, "bad sizes n_q=%d n_cur=%d Hq=%d", n_q, n_cur, Hq);
    if (Hq % L.Hkv != 0) return set_error(KV_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, L.Hkv);
    if (n_cur > 0 && (!Kcur || !Vcur)) return set_error(KV_ERR_INVALID_ARG, "Kcur/Vcur NULL with n_cur > 0");
    if (!aligned16(Q) || !aligned16(out) || (n_cur > 0 && (!aligned16(Kcur) || !aligned16(Vcur))))
        return set_error(KV_ERR_ALIGNMENT, "Q, Kcur, Vcur and out must be 16-byte aligned");
    if (dtype < KV_F32 || dtype > KV_BF16) return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (L.kind == KV_MIXED && (int)dtype != L.raw_dtype)
        return set_error(KV_ERR_UNSUPPORTED, "MIXED cache: I/O dtype must equal raw_dtype");
    const kv_attn_opts dflt = {0.0f, KV_JENSEN_OFF, 0, 0, 0, KV_PATH_AUTO};
    const kv_attn_opts* o = opts ? opts : &dflt;
    if (o->jensen < KV_JENSEN_OFF || o->jensen > KV_JENSEN_ISOTROPIC) return set_error(KV_ERR_INVALID_ARG, "bad jensen mode");
    if (o->psac && (L.kind != KV_CODEBOOK2 || L.psac_rank == 0 || !cache->psac_u))
        return set_error(KV_ERR_INVALID_ARG, "psac needs a CODEBOOK2 cache with psac_rank > 0 and a basis");
    if (L.kind == KV_CODEBOOK2 && cache->resid_var && o->jensen == KV_JENSEN_EXACT)
        return set_error(KV_ERR_UNSUPPORTED, "the EXACT Jensen form is not defined for codebook keys");
    const float tau = o->scale != 0.0f ? o->scale : 1.0f / sqrtf((float)L.d);
    const int path = pick_path(cache, dtype, n_q, Hq, o);
    const int sp = pick_splits(cache, path, n_q, n_cur, Hq, o);
    size_t need = 0;
    if (path == KV_PATH_DECODE) need = decode_workspace(cache, Hq, sp);
    else if (path == KV_PATH_TC || path == KV_PATH_TC_SINGLE) need = tc_workspace(cache, n_q, Hq, sp);
    else need = simt_workspace(cache, n_q, Hq, sp);
    if (!workspace || ws_bytes < need)
        return set_error(KV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, ws_bytes);
    if (!aligned16(workspace)) return set_error(KV_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    kv_status r;
    switch (path) {
        case KV_PATH_SIMT:
            r = launch_attn_simt(Q, Kcur, Vcur, dtype, n_q, n_cur, Hq, cache, tau, o->jensen, o->psac, sp, out,
                                 o->out_f32, lse, workspace, st);
            break;
        case KV_PATH_DECODE:
            if (!decode_supported(cache, dtype, n_q, Hq))
                return set_error(KV_ERR_UNSUPPORTED, "decode path: needs n_q == 1, f16/bf16, d in {64,128}, "
                                 "UNIFORM/MIXED cache and at most 16 query heads per kv head");
            if (o->psac) return set_error(KV_ERR_UNSUPPORTED, "decode path has no PSAC term");
            // automatic splits: one wave of resident CTAs, some streams one split fewer
            r = launch_attn_decode(Q, Kcur, Vcur, dtype, n_cur, Hq, cache, tau, o->jensen, sp,
                                   o->num_splits > 0 ? 0 : decode_auto_ctas(cache, Hq, sp), out, o->out_f32, lse,
                                   workspace, st);
            break;
        case KV_PATH_TC:
        case KV_PATH_TC_SINGLE: {
            const char* why = "";
            if (!tc_supported(cache, dtype, n_q, Hq, &why))
                return set_error(KV_ERR_UNSUPPORTED, "tensor-core path: %s", why);
            r = launch_attn_tc(Q, Kcur, Vcur, n_q, n_cur, Hq, cache, tau, o->jensen, o->psac, sp, out, o->out_f32,
                               lse, workspace, path == KV_PATH_TC, st);
            break;
        }
        default:
            return set_error(KV_ERR_INVALID_ARG, "unknown path %d", path);
    }
    // debugging: wait for the call and report its status words at once
    if (r == KV_OK && getenv("BITKV_DEBUG_SYNC")) r = read_status(workspace, st);
    return r;
}

kv_status kv_attention_status(const void* workspace, void* stream) {
    if (!workspace) return set_error(KV_ERR_INVALID_ARG, "workspace is NULL");
    return read_status(workspace, static_cast<cudaStream_t>(stream));
}

kv_status kv_window_plan(const float* sim, int n_windows, const kv_thresholds* th, int8_t* bits_out,
                         int32_t* perm_out) {
    if (n_windows < 0) return set_error(KV_ERR_INVALID_ARG, "n_windows < 0");
    if (n_windows == 0) return KV_OK;
    if (!sim || !bits_out) return set_error(KV_ERR_INVALID_ARG, "sim or bits_out is NULL");
    const double f16 = th ? th->frac_fp16 : 0.2, f4 = th ? th->frac_int4 : 0.3;
    const int force_first = th ? th->force_first : 1;
    if (!(f16 >= 0.0) || !(f4 >= 0.0) || f16 + f4 > 1.0 + 1e-12)
        return set_error(KV_ERR_INVALID_ARG, "fractions must be >= 0 with sum <= 1");
    for (int w = 0; w < n_windows; ++w)
        if (std::isnan(sim[w])) return set_error(KV_ERR_INVALID_ARG, "sim[%d] is NaN", w);
    const int first = force_first ? 1 : 0;
    std::vector<int> order;
    for (int w = first; w < n_windows; ++w) order.push_back(w);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (sim[a] != sim[b]) return sim[a] > sim[b];
        return a < b;
    });
    const int n = (int)order.size();
    const int n16 = (int)std::floor(f16 * (double)n);
    const int nhi = std::max(n16, (int)std::floor((f16 + f4) * (double)n));
    for (int w = 0; w < n_windows; ++w) bits_out[w] = 2;
    if (force_first) bits_out[0] = 16;
    for (int rk = 0; rk < n; ++rk) bits_out[order[rk]] = rk < n16 ? 16 : (rk < nhi ? 4 : 2);
    if (perm_out) {
        int k = 0;
        for (int cls : {16, 4, 2})
            for (int w = 0; w < n_windows; ++w)
                if (bits_out[w] == cls) perm_out[k++] = w;
    }
    return KV_OK;
}

size_t kv_codebook_workspace(const kv_layout* L, int n_tokens) { return L ? codebook_ws_bytes(L, n_tokens) : 0; }

kv_status kv_codebook_fit(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, int iters, const void* Qhist,
                          int n_hist, float* weights_out, void* workspace, size_t ws_bytes, void* stream) {
    AbiRange nvtx_range("kv_codebook_fit");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (cache->layout.kind != KV_CODEBOOK2) return set_error(KV_ERR_INVALID_ARG, "cache is not CODEBOOK2");
    if (!K || !cache->centroids) return set_error(KV_ERR_INVALID_ARG, "K or centroids NULL");
    if (n_tokens <= 0 || iters < 0) return set_error(KV_ERR_INVALID_ARG, "n_tokens must be > 0, iters >= 0");
    if (Qhist && (n_hist <= 0 || !weights_out)) return set_error(KV_ERR_INVALID_ARG, "Qhist needs n_hist > 0 and weights_out");
    const size_t need = codebook_ws_bytes(&cache->layout, n_tokens);
    if (need && (!workspace || ws_bytes < need))
        return set_error(KV_ERR_WORKSPACE, "codebook workspace of %zu bytes needed, %zu given", need, ws_bytes);
    return launch_codebook_fit(K, dtype, n_tokens, cache, iters, Qhist, n_hist, weights_out, 0, workspace,
                               static_cast<cudaStream_t>(stream));
}

kv_status kv_codebook_fit_range(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, int iters,
                                const void* Qhist, int n_hist, float* weights_out, void* stream) {
    AbiRange nvtx_range("kv_codebook_fit_range");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (cache->layout.kind != KV_CODEBOOK2) return set_error(KV_ERR_INVALID_ARG, "cache is not CODEBOOK2");
    if (!K || !cache->centroids) return set_error(KV_ERR_INVALID_ARG, "K or centroids NULL");
    if (n_tokens <= 0 || iters < 0) return set_error(KV_ERR_INVALID_ARG, "n_tokens must be > 0, iters >= 0");
    if (!Qhist || n_hist <= 0 || !weights_out)
        return set_error(KV_ERR_INVALID_ARG, "the residual-range fit needs Qhist, n_hist > 0 and weights_out");
    if (dtype < KV_F32 || dtype > KV_BF16) return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    return launch_codebook_fit(K, dtype, n_tokens, cache, iters, Qhist, n_hist, weights_out, 1, nullptr,
                               static_cast<cudaStream_t>(stream));
}

kv_status kv_codebook_residual_var(const void* K, kv_dtype dtype, int n_tokens, kv_cache* cache, void* stream) {
    AbiRange nvtx_range("kv_codebook_residual_var");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (cache->layout.kind != KV_CODEBOOK2) return set_error(KV_ERR_INVALID_ARG, "cache is not CODEBOOK2");
    if (!K || !cache->centroids || !cache->resid_var)
        return set_error(KV_ERR_INVALID_ARG, "K, centroids or resid_var NULL");
    if (n_tokens <= 0) return set_error(KV_ERR_INVALID_ARG, "n_tokens must be > 0");
    if (dtype < KV_F32 || dtype > KV_BF16) return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    return launch_residual_var(K, dtype, n_tokens, cache, static_cast<cudaStream_t>(stream));
}

size_t kv_psac_workspace(const kv_layout* L) { return L ? psac_ws_bytes(L) : 0; }

kv_status kv_psac_basis(const void* Qhist, kv_dtype dtype, int n_hist, kv_cache* cache, float* eigvals_out,
                        void* workspace, size_t ws_bytes, void* stream) {
    AbiRange nvtx_range("kv_psac_basis");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (cache->layout.kind != KV_CODEBOOK2 || cache->layout.psac_rank <= 0 || !cache->psac_u)
        return set_error(KV_ERR_INVALID_ARG, "PSAC basis needs a CODEBOOK2 cache with psac_rank > 0 and psac_u");
    if (!Qhist || n_hist <= 0) return set_error(KV_ERR_INVALID_ARG, "Qhist NULL or n_hist <= 0");
    const size_t need = psac_ws_bytes(&cache->layout);
    if (need && (!workspace || ws_bytes < need))
        return set_error(KV_ERR_WORKSPACE, "PSAC workspace of %zu bytes needed, %zu given", need, ws_bytes);
    return launch_psac_basis(Qhist, dtype, n_hist, cache, eigvals_out, workspace, static_cast<cudaStream_t>(stream));
}

kv_status kv_debug_operands(const kv_cache* cache, int path, void* K_out, void* V_out, void* stream) {
    AbiRange nvtx_range("kv_debug_operands");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (!K_out || !V_out) return set_error(KV_ERR_INVALID_ARG, "K_out or V_out is NULL");
    if (!aligned16(K_out) || !aligned16(V_out)) return set_error(KV_ERR_ALIGNMENT, "K_out and V_out must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (path == KV_PATH_TC) return launch_tc_operands(cache, K_out, V_out, st);
    if (path == KV_PATH_DECODE) return launch_dec_operands(cache, K_out, V_out, st);
    return set_error(KV_ERR_INVALID_ARG, "kv_debug_operands: path must be KV_PATH_TC or KV_PATH_DECODE");
}

kv_status kv_dequantize(const kv_cache* cache, float* K_out, float* V_out, void* stream) {
    AbiRange nvtx_range("kv_dequantize");
    kv_status s = check_cache(cache);
    if (s != KV_OK) return s;
    if (!K_out || !V_out) return set_error(KV_ERR_INVALID_ARG, "K_out or V_out is NULL");
    return launch_dequant(cache, K_out, V_out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
