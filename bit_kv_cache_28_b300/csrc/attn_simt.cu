// CUDA-core attention over any cache kind, with split-KV partials and the
// log-sum-exp merge.  It is the exact-fp32 path: every operand (queries, the
// dequantised cache entries fmaf(code, s, z), the current chunk) enters the
// products as the fp32 value it is, and sums run in fp32.  It serves every dtype
// and the shapes the tensor-core kernel does not take.
//
// "Quantized Keys Steal Attention" (abstract): queries of the current chunk
// attend to the cached chunks and to the current, unquantised chunk; the
// Jensen correction is computed on the fly from the cached keys' step sizes and
// the query.  "QuantWM" (Innovations 3): PSAC adds a low-rank key correction
// along the query subspace.
//
// CTA = 32 queries x 128 threads; a row's 4 threads split the 32 keys of a
// tile (logits) and the d channels (output, interleaved so shared-memory
// accesses do not conflict).  A tile is one cache block or 32 current tokens.
#include "common.cuh"

namespace bitkv {

namespace {

constexpr int kSQ = 32;
constexpr int kSK = 32;
constexpr int kSimtThreads = 128;

struct SimtSmem {
    // offsets in floats
    int qs, ks, vs, ss, sk, uq, cq, stg;
    int total;
};

// A staged cache block: up to the size of a 16-bit block (32 tokens x d x 2 bytes x K and V),
// the largest block of any class at head dim d.
__host__ __device__ constexpr int simt_stage_bytes(int d) { return kSK * d * 2 * 2; }

__host__ __device__ inline SimtSmem simt_smem(int d, int r) {
    SimtSmem s;
    const int ld = d + 1;
    s.qs = 0;
    s.ks = s.qs + kSQ * ld;
    s.vs = s.ks + kSK * ld;
    s.ss = s.vs + kSK * ld;
    s.sk = s.ss + kSQ * (kSK + 1);
    s.uq = s.sk + d;
    s.cq = s.uq + kSQ * (r > 0 ? r : 1);
    s.stg = (s.cq + kSK * (r > 0 ? r : 1) + 3) & ~3;   // 16-byte aligned
    s.total = s.stg + simt_stage_bytes(d) / 4;
    return s;
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads)
attn_simt_kernel(const T* __restrict__ Q, const T* __restrict__ Kcur, const T* __restrict__ Vcur, int n_q, int n_cur,
                 int Hq, DevCache c, float tau, int jensen, int use_psac, int n_splits, int units_cache,
                 int units_total, void* __restrict__ out, int out_f32, float* __restrict__ lse,
                 float* __restrict__ ws_o, float2* __restrict__ ws_ml) {
    extern __shared__ float smem[];
    const int n_qt = (n_q + kSQ - 1) / kSQ;
    const int qt = blockIdx.x % n_qt, split = blockIdx.x / n_qt;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int grp = Hq / c.Hkv, h = hq / grp;
    const int tid = threadIdx.x, row = tid >> 2, part = tid & 3;
    const int q0 = qt * kSQ;
    constexpr int ld = D + 1;
    const int r = use_psac ? c.r : 0;
    const SimtSmem L = simt_smem(D, c.r);
    float* Qs = smem + L.qs;
    float* Ks = smem + L.ks;
    float* Vs = smem + L.vs;
    float* Ss = smem + L.ss;
    float* Sk = smem + L.sk;
    float* Uq = smem + L.uq;
    float* Cq = smem + L.cq;
    uint4* stg = reinterpret_cast<uint4*>(smem + L.stg);

    // loops with a fixed trip count and read-only loads, so that a thread's loads are all in
    // flight before their results are stored
    const long long qbase = (((long long)b * Hq + hq) * n_q) * D;
#pragma unroll 8
    for (int it = 0; it < kSQ * D / kSimtThreads; ++it) {
        const int e = tid + it * kSimtThreads, i = e / D, ch = e % D;
        Qs[i * ld + ch] = (q0 + i < n_q) ? to_f32<T>(__ldg(Q + qbase + (long long)(q0 + i) * D + ch)) : 0.0f;
    }
    __syncthreads();
    if (r > 0) {
        const float* U = c.psac_u + ((long long)b * c.Hkv + h) * D * r;
        for (int e = tid; e < kSQ * r; e += kSimtThreads) {
            const int i = e / r, jj = e % r;
            float a = 0.0f;
            for (int ch = 0; ch < D; ++ch) a = fmaf(Qs[i * ld + ch], U[ch * r + jj], a);
            Uq[i * r + jj] = a;
        }
    }

    // codebook keys with residual variances: the row's Jensen term (tau^2/2) sum_c q'_c^2 v_c
    // (ISOTROPIC: |q'|^2 mean_c v_c), q' = q - U (U^T q) with the PSAC term on, the same
    // for every cached key; the 4 threads of a row split the channels
    float cb_delta = 0.0f;
    if (c.kind == KV_CODEBOOK2 && c.resid_var && jensen != KV_JENSEN_OFF) {
        __syncthreads();                   // U^T q of the rows is in shared memory
        const float* vv = c.resid_var + ((long long)b * c.Hkv + h) * D;
        const float* U = r > 0 ? c.psac_u + ((long long)b * c.Hkv + h) * D * r : nullptr;
        float acc = 0.0f, qn = 0.0f, vs = 0.0f;
        for (int ch = part; ch < D; ch += 4) {
            float qc = Qs[row * ld + ch];
            for (int jj = 0; jj < r; ++jj) qc = fmaf(-U[ch * r + jj], Uq[row * r + jj], qc);
            const float var = vv[ch];
            acc = fmaf(qc * qc, var, acc);
            qn = fmaf(qc, qc, qn);
            vs += var;
        }
#pragma unroll
        for (int m = 1; m < 4; m <<= 1) {
            acc += __shfl_xor_sync(0xffffffffu, acc, m);
            qn += __shfl_xor_sync(0xffffffffu, qn, m);
            vs += __shfl_xor_sync(0xffffffffu, vs, m);
        }
        cb_delta = 0.5f * tau * tau * (jensen == KV_JENSEN_ISOTROPIC ? qn * (vs * (1.0f / D)) : acc);
    }

    float m_run = -INFINITY, l_run = 0.0f;
    float o[D / 4];
#pragma unroll
    for (int i = 0; i < D / 4; ++i) o[i] = 0.0f;

    const int u0 = (int)((long long)split * units_total / n_splits);
    const int u1 = (int)((long long)(split + 1) * units_total / n_splits);
    const float* cent = c.centroids ? c.centroids + ((long long)b * c.Hkv + h) * D * 4 : nullptr;

    for (int u = u0; u < u1; ++u) {
        __syncthreads();
        int len, quantised = 0, has_coeff = 0, codebook = 0;
        if (u < units_cache) {
            int seg = 0, i = u;
            while (i >= c.n_blocks[seg]) {
                i -= c.n_blocks[seg];
                ++seg;
            }
            const long long gi = (long long)b * c.cap_total + c.seg_base[seg] + i;
            len = c.blk_len[gi];
            const unsigned char* blk = block_ptr(c, b, h, seg, i);
            const int cls = seg_class(c.kind, seg);
            // the packed block into shared memory: one coalesced pass of 16-byte loads, all
            // issued before the stores (the entries are then decoded from the staged copy)
            constexpr int kPass = simt_stage_bytes(D) / (16 * kSimtThreads);
            const int n16 = (int)(c.block_bytes[seg] >> 4);
            if (n16 <= kPass * kSimtThreads) {
                const uint4* src = reinterpret_cast<const uint4*>(blk);
                uint4 tmp[kPass];
#pragma unroll
                for (int k = 0; k < kPass; ++k) {
                    const int x = tid + k * kSimtThreads;
                    tmp[k] = x < n16 ? __ldg(src + x) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < kPass; ++k) {
                    const int x = tid + k * kSimtThreads;
                    if (x < n16) stg[x] = tmp[k];
                }
                __syncthreads();
                blk = reinterpret_cast<const unsigned char*>(stg);
            }
            for (int e = tid; e < kSK * D; e += kSimtThreads) {
                const int t = e / D, ch = e % D;
                const float2 kv =
                    t < len ? block_entry(cls, blk, D, c.raw_dtype, c.meta16, cent, t, ch) : make_float2(0.f, 0.f);
                Ks[t * ld + ch] = kv.x;     // the exact dequantised entries
                Vs[t * ld + ch] = kv.y;
            }
            if (cls == CLS_INT2 || cls == CLS_INT4) {
                quantised = 1;
                const unsigned char* km = blk + int_offsets(D, cls == CLS_INT4 ? 4 : 2, c.meta16).km;
                for (int ch = tid; ch < D; ch += kSimtThreads) Sk[ch] = meta_at(km, ch, c.meta16).x;
            }
            codebook = cls == CLS_CB2;
            if (cls == CLS_CB2 && r > 0) {
                has_coeff = 1;
                const __half* kq = reinterpret_cast<const __half*>(blk + cb_offsets(D).kq);
                for (int e = tid; e < kSK * r; e += kSimtThreads) {
                    const int t = e / r, jj = e % r;
                    Cq[t * r + jj] = __half2float(kq[t * c.rp + jj]);
                }
            }
        } else {
            const int t0 = (u - units_cache) * kSK;
            len = min(kSK, n_cur - t0);
            const long long kb = (((long long)b * c.Hkv + h) * n_cur + t0) * D;
#pragma unroll 8
            for (int it = 0; it < kSK * D / kSimtThreads; ++it) {
                const int e = tid + it * kSimtThreads, t = e / D, ch = e % D;
                Ks[t * ld + ch] = t < len ? to_f32<T>(__ldg(Kcur + kb + e)) : 0.0f;
                Vs[t * ld + ch] = t < len ? to_f32<T>(__ldg(Vcur + kb + e)) : 0.0f;
            }
        }
        __syncthreads();

        // Jensen correction of this block for this row
        float delta = codebook ? cb_delta : 0.0f;
        if (quantised && jensen != KV_JENSEN_OFF) {
            float qn2 = 0.0f, ss2 = 0.0f;    // ISOTROPIC: |q|^2 and sum_c s_c^2
            for (int ch = part; ch < D; ch += 4) {
                const float q = Qs[row * ld + ch], s = Sk[ch];
                if (jensen == KV_JENSEN_TAYLOR2) delta = fmaf(q * q, s * s, delta);
                else if (jensen == KV_JENSEN_ISOTROPIC) {
                    qn2 = fmaf(q, q, qn2);
                    ss2 = fmaf(s, s, ss2);
                } else delta += log_sinhc(0.5f * tau * q * s);
            }
            if (jensen == KV_JENSEN_ISOTROPIC) {
                qn2 += __shfl_xor_sync(0xffffffffu, qn2, 1);
                qn2 += __shfl_xor_sync(0xffffffffu, qn2, 2);
                ss2 += __shfl_xor_sync(0xffffffffu, ss2, 1);
                ss2 += __shfl_xor_sync(0xffffffffu, ss2, 2);
                delta = tau * tau * (1.0f / 24.0f) * qn2 * (ss2 * (1.0f / D));
            } else {
                delta += __shfl_xor_sync(0xffffffffu, delta, 1);
                delta += __shfl_xor_sync(0xffffffffu, delta, 2);
                if (jensen == KV_JENSEN_TAYLOR2) delta *= tau * tau * (1.0f / 24.0f);
            }
        }
        float lg[kSK / 4];
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < kSK / 4; ++i) {
            const int k = part + 4 * i;
            float a = 0.0f;
#pragma unroll 8
            for (int ch = 0; ch < D; ++ch) a = fmaf(Qs[row * ld + ch], Ks[k * ld + ch], a);
            float l = tau * a - delta;
            if (has_coeff) {
                float p = 0.0f;
                for (int jj = 0; jj < r; ++jj) p = fmaf(Uq[row * r + jj], Cq[k * r + jj], p);
                l = fmaf(tau, p, l);
            }
            if (k >= len) l = -INFINITY;
            lg[i] = l;
            tmax = fmaxf(tmax, l);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);
        const float m_use = m_new == -INFINITY ? 0.0f : m_new;   // no valid key yet: every p is 0
        const float corr = expf(m_run - m_use);
        float psum = 0.0f;
#pragma unroll
        for (int i = 0; i < kSK / 4; ++i) {
            const float p = expf(lg[i] - m_use);
            Ss[row * (kSK + 1) + part + 4 * i] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l_run = l_run * corr + psum;
        m_run = m_new;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < D / 4; ++i) o[i] *= corr;
        for (int k = 0; k < kSK; ++k) {
            const float p = Ss[row * (kSK + 1) + k];
#pragma unroll
            for (int i = 0; i < D / 4; ++i) o[i] = fmaf(p, Vs[k * ld + 4 * i + part], o[i]);
        }
        __syncwarp();
    }

    const int qi = q0 + row;
    if (qi >= n_q) return;
    const long long orow = ((long long)b * Hq + hq) * n_q + qi;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    if (n_splits == 1) {
        for (int i = 0; i < D / 4; ++i) {
            const float v = o[i] * inv;
            if (out_f32) static_cast<float*>(out)[orow * D + 4 * i + part] = v;
            else static_cast<T*>(out)[orow * D + 4 * i + part] = from_f32<T>(v);
        }
        if (lse && part == 0) lse[orow] = m_run + logf(l_run);
    } else {
        const long long rows = (long long)c.B * Hq * n_q;
        float* wo = ws_o + ((long long)split * rows + orow) * D;
        for (int i = 0; i < D / 4; ++i) wo[4 * i + part] = o[i] * inv;
        if (part == 0) ws_ml[(long long)split * rows + orow] = make_float2(m_run, l_run);
    }
}

// Merge split partials: m = max m_p, l = sum l_p e^{m_p - m}, o = sum l_p e^{m_p - m} o_p / l.
// One warp per row: the split weights are reduced across lanes, then each lane
// combines 4 channels (128-bit loads) per pass over the splits.
constexpr int kMergeRows = 8;   // rows (warps) per CTA

template <typename T>
__global__ void __launch_bounds__(32 * kMergeRows)
lse_merge_kernel(const float* __restrict__ ws_o, const float2* __restrict__ ws_ml, int n_splits, long long rows, int d,
                 void* __restrict__ out, int out_f32, float* __restrict__ lse) {
    const long long row = (long long)blockIdx.x * kMergeRows + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float m = -INFINITY;
    for (int p = lane; p < n_splits; p += 32) {
        const float2 ml = ws_ml[p * rows + row];
        if (ml.y > 0.0f) m = fmaxf(m, ml.x);
    }
    m = warp_max(m);
    float l = 0.0f;
    for (int p = lane; p < n_splits; p += 32) {
        const float2 ml = ws_ml[p * rows + row];
        if (ml.y > 0.0f) l += ml.y * expf(ml.x - m);
    }
    l = warp_sum(l);
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    for (int c4 = lane; c4 < d / 4; c4 += 32) {
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int p = 0; p < n_splits; ++p) {
            const float2 ml = ws_ml[p * rows + row];
            if (ml.y > 0.0f) {
                const float w = ml.y * expf(ml.x - m);
                const float4 o = reinterpret_cast<const float4*>(ws_o + (p * rows + row) * d)[c4];
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
            }
        }
        const float v[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
        if (out_f32) {
            reinterpret_cast<float4*>(static_cast<float*>(out) + row * d)[c4] = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            T* o = static_cast<T*>(out) + row * d + 4 * c4;
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = from_f32<T>(v[k]);
        }
    }
    if (lse && lane == 0) lse[row] = m + logf(l);
}

}  // namespace

static unsigned merge_grid(long long rows) { return (unsigned)((rows + kMergeRows - 1) / kMergeRows); }

kv_status launch_lse_merge(kv_dtype dt, const float* ws_o, const float2* ws_ml, int n_splits, long long rows, int d,
                           void* out, int out_f32, float* lse, cudaStream_t st) {
    switch (dt) {
        case KV_F32:
            lse_merge_kernel<float><<<merge_grid(rows), 32 * kMergeRows, 0, st>>>(ws_o, ws_ml, n_splits, rows, d, out,
                                                                                 out_f32, lse);
            break;
        case KV_F16:
            lse_merge_kernel<__half><<<merge_grid(rows), 32 * kMergeRows, 0, st>>>(ws_o, ws_ml, n_splits, rows, d, out,
                                                                                  out_f32, lse);
            break;
        case KV_BF16:
            lse_merge_kernel<__nv_bfloat16><<<merge_grid(rows), 32 * kMergeRows, 0, st>>>(ws_o, ws_ml, n_splits, rows,
                                                                                         d, out, out_f32, lse);
            break;
    }
    return check_launch("lse_merge_kernel");
}

int simt_units_cache(const kv_cache* c) { return c->n_blocks[0] + c->n_blocks[1] + c->n_blocks[2]; }

size_t simt_smem_bytes(int d, int r) { return simt_smem(d, r).total * sizeof(float); }

template <typename T, int D>
static void launch_simt_td(const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq, const DevCache& c,
                           float tau, int jensen, int psac, int n_splits, int uc, int ut, void* out, int out_f32,
                           float* lse, float* ws_o, float2* ws_ml, cudaStream_t st) {
    const size_t sm = simt_smem_bytes(D, c.r);
    // a refusal leaves the limit unset; the launch then fails and the caller reports it
    (void)set_smem_limit(reinterpret_cast<const void*>(attn_simt_kernel<T, D>), 200 * 1024, "attn_simt_kernel");
    const int n_qt = (n_q + kSQ - 1) / kSQ;
    dim3 grid(n_qt * n_splits, Hq, c.B);
    attn_simt_kernel<T, D><<<grid, kSimtThreads, sm, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(Kc), static_cast<const T*>(Vc), n_q, n_cur, Hq, c, tau, jensen,
        psac, n_splits, uc, ut, out, out_f32, lse, ws_o, ws_ml);
}

template <typename T>
static kv_status launch_simt_t(const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                               const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out,
                               int out_f32, float* lse, void* ws, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    const int uc = simt_units_cache(cache);
    const int ut = uc + (n_cur + kSK - 1) / kSK;
    const long long rows = (long long)c.B * Hq * n_q;
    // the status header stays zero: this kernel has no bounded waits and no fp16 operands
    const kv_status sc = clear_device(ws, kStatusBytes, st, "attn_simt_kernel");
    if (sc != KV_OK) return sc;
    float* ws_o = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kStatusBytes);
    float2* ws_ml = reinterpret_cast<float2*>(ws_o + (n_splits > 1 ? (long long)n_splits * rows * c.d : 0));
    switch (c.d) {
        case 32: launch_simt_td<T, 32>(Q, Kc, Vc, n_q, n_cur, Hq, c, tau, jensen, psac, n_splits, uc, ut, out, out_f32, lse, ws_o, ws_ml, st); break;
        case 64: launch_simt_td<T, 64>(Q, Kc, Vc, n_q, n_cur, Hq, c, tau, jensen, psac, n_splits, uc, ut, out, out_f32, lse, ws_o, ws_ml, st); break;
        case 128: launch_simt_td<T, 128>(Q, Kc, Vc, n_q, n_cur, Hq, c, tau, jensen, psac, n_splits, uc, ut, out, out_f32, lse, ws_o, ws_ml, st); break;
        case 256: launch_simt_td<T, 256>(Q, Kc, Vc, n_q, n_cur, Hq, c, tau, jensen, psac, n_splits, uc, ut, out, out_f32, lse, ws_o, ws_ml, st); break;
        default: return set_error(KV_ERR_UNSUPPORTED, "SIMT attention: d=%d not in {32,64,128,256}", c.d);
    }
    kv_status s = check_launch("attn_simt_kernel");
    if (s != KV_OK || n_splits == 1) return s;
    lse_merge_kernel<T><<<merge_grid(rows), 32 * kMergeRows, 0, st>>>(ws_o, ws_ml, n_splits, rows, c.d, out, out_f32,
                                                                      lse);
    return check_launch("lse_merge_kernel");
}

kv_status launch_attn_simt(const void* Q, const void* Kc, const void* Vc, kv_dtype dt, int n_q, int n_cur, int Hq,
                           const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out,
                           int out_f32, float* lse, void* ws, cudaStream_t st) {
    switch (dt) {
        case KV_F32: return launch_simt_t<float>(Q, Kc, Vc, n_q, n_cur, Hq, cache, tau, jensen, psac, n_splits, out, out_f32, lse, ws, st);
        case KV_F16: return launch_simt_t<__half>(Q, Kc, Vc, n_q, n_cur, Hq, cache, tau, jensen, psac, n_splits, out, out_f32, lse, ws, st);
        case KV_BF16: return launch_simt_t<__nv_bfloat16>(Q, Kc, Vc, n_q, n_cur, Hq, cache, tau, jensen, psac, n_splits, out, out_f32, lse, ws, st);
    }
    return set_error(KV_ERR_INVALID_ARG, "unknown dtype");
}

size_t simt_workspace(const kv_cache* cache, int n_q, int Hq, int n_splits) {
    if (n_splits <= 1) return kStatusBytes;
    const long long rows = (long long)cache->layout.B * Hq * n_q;
    return kStatusBytes + (size_t)n_splits * rows * (cache->layout.d * sizeof(float) + sizeof(float2));
}

}  // namespace bitkv
