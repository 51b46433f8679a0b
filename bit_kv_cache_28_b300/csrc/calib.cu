// Calibration kernels of the codebook cache: QSAC key centroids and the PSAC basis.
//
// "QuantWM" (Innovations 2, Methodology): INT2 key centroids chosen per channel
// by quantisation-sensitivity-aware clustering.  Read as a per-(head, channel)
// 1-D Lloyd k-means with 4 centroids: quantile initialisation x_(floor((2k+1)n/8))
// of the sorted values, then `iters` rounds of nearest-centroid assignment by the
// fp64 distance |x - mu_k| (ties to the lower k) and mu_k = (member sum) / n_k in
// fp64, an empty cluster keeping its centroid.  The per-channel sensitivity
// weight mean_t q_c^2 of the historical queries is a constant factor inside one
// channel's 1-D problem and changes no centroid; it is computed and returned.
// Member sums of 16-bit inputs are exact in fp64 at these sizes, so the block
// reduction order does not matter.
//
// QSAC with residual ranges (the pages: the clustering weighs the queries'
// sensitivity together with the range of the residuals, protecting the channels
// that matter more): given the weights, channel c of a (b, h) gets rho_c = w_c / max w
// (fp64 of the fp32 weights) and each update moves the cluster's mean towards its
// mid-range, mu_k = mean_k + rho_c (mid_k - mean_k), mid_k = (min_k + max_k) / 2,
// every fp64 operation rounded once in that order (no contraction), so the centroids
// match the oracle's bit for bit.  rho = 0 is Lloyd.
//
// "QuantWM" (Innovations 3): PSAC compensates the remaining key error along the
// dominant subspace of the queries.  U = the top-r eigenvectors of the uncentred
// second moment C = (1/n) sum_t q_t q_t^T of the historical queries, eigenvalues
// descending, each column signed so its largest-magnitude entry is positive.
// C is accumulated in fp64; its eigenvectors come from a cyclic Jacobi method in
// fp64 whose rotations are applied in parallel rounds of d/2 disjoint index pairs
// (a round-robin tournament ordering), with the matrix in shared memory and the
// accumulated rotations in the workspace.
#include <cmath>
#include <cstdio>

#include "common.cuh"

namespace bitkv {

namespace {

constexpr int kCbThreads = 256;
constexpr int kJThreads = 256;
constexpr int kMaxCbTokens = 32768;   // values per channel sorted in shared memory
constexpr int kMaxSweeps = 40;

template <typename T> __device__ __forceinline__ float load_f32(const T* p) { return to_f32<T>(*p); }

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One CTA per (channel, kv head, batch row).  w (nullable): the fp32 sensitivity
// weights [B][Hkv][d] for the residual-range update; NULL for Lloyd.
template <typename T>
__global__ void __launch_bounds__(kCbThreads)
codebook_fit_kernel(const T* __restrict__ K, int n, int npow2, int d, int Hkv, int iters, const float* __restrict__ w,
                    float* __restrict__ cent) {
    extern __shared__ float xs[];                   // [npow2] values, sorted in place
    __shared__ double s_sum[kCbThreads / 32][4];
    __shared__ int s_cnt[kCbThreads / 32][4];
    __shared__ float s_mn[kCbThreads / 32][4], s_mx[kCbThreads / 32][4];
    __shared__ double s_mu[4];
    __shared__ float s_wmax[kCbThreads / 32];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    double rho = 0.0;
    if (w) {
        const float* wb = w + ((long long)b * Hkv + h) * d;
        float m = 0.0f;
        for (int e = tid; e < d; e += kCbThreads) m = fmaxf(m, wb[e]);
        m = warp_max(m);
        if (lane == 0) s_wmax[warp] = m;
        __syncthreads();
        float wm = 0.0f;
        for (int q = 0; q < kCbThreads / 32; ++q) wm = fmaxf(wm, s_wmax[q]);
        rho = wm > 0.0f ? (double)wb[c] / (double)wm : 0.0;
    }
    const T* src = K + ((long long)b * Hkv + h) * n * d + c;
    for (int t = tid; t < npow2; t += kCbThreads) xs[t] = t < n ? load_f32(src + (long long)t * d) : INFINITY;
    __syncthreads();
    // bitonic sort, ascending (padding +inf sorts to the end)
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow2; i += kCbThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const float a = xs[i], bq = xs[l];
                    const bool up = (i & k) == 0;
                    if ((a > bq) == up) {
                        xs[i] = bq;
                        xs[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (tid < 4) s_mu[tid] = (double)xs[((long long)(2 * tid + 1) * n) / 8];
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
        const double mu0 = s_mu[0], mu1 = s_mu[1], mu2 = s_mu[2], mu3 = s_mu[3];
        double sum[4] = {0.0, 0.0, 0.0, 0.0};
        int cnt[4] = {0, 0, 0, 0};
        float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        for (int t = tid; t < n; t += kCbThreads) {
            const float xf = xs[t];
            const double x = xf;
            double best = fabs(x - mu0);
            int k = 0;
            const double d1 = fabs(x - mu1), d2 = fabs(x - mu2), d3 = fabs(x - mu3);
            if (d1 < best) { best = d1; k = 1; }
            if (d2 < best) { best = d2; k = 2; }
            if (d3 < best) { best = d3; k = 3; }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q == k) {
                    sum[q] += x;
                    cnt[q] += 1;
                    mn[q] = fminf(mn[q], xf);
                    mx[q] = fmaxf(mx[q], xf);
                }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            sum[q] = warp_sum_d(sum[q]);
            cnt[q] = warp_sum_i(cnt[q]);
            mn[q] = warp_min(mn[q]);
            mx[q] = warp_max(mx[q]);
        }
        if (lane == 0)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                s_sum[warp][q] = sum[q];
                s_cnt[warp][q] = cnt[q];
                s_mn[warp][q] = mn[q];
                s_mx[warp][q] = mx[q];
            }
        __syncthreads();
        if (tid < 4) {
            double sm = 0.0;
            int cn = 0;
            float lo = INFINITY, hi = -INFINITY;
            for (int q = 0; q < kCbThreads / 32; ++q) {
                sm += s_sum[q][tid];
                cn += s_cnt[q][tid];
                lo = fminf(lo, s_mn[q][tid]);
                hi = fmaxf(hi, s_mx[q][tid]);
            }
            if (cn > 0) {
                const double mean = sm / (double)cn;
                if (w) {
                    const double mid = __dmul_rn(__dadd_rn((double)lo, (double)hi), 0.5);
                    s_mu[tid] = __dadd_rn(mean, __dmul_rn(rho, __dsub_rn(mid, mean)));
                } else {
                    s_mu[tid] = mean;
                }
            }
        }
        __syncthreads();
    }
    if (tid < 4) cent[(((long long)b * Hkv + h) * d + c) * 4 + tid] = (float)s_mu[tid];
}

// Sensitivity weight w_c = mean_t q_{t,c}^2 of the historical queries; one thread per (b, h, c).
template <typename T>
__global__ void sensitivity_kernel(const T* __restrict__ Qh, int n_hist, int d, long long total, float* __restrict__ w) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const long long bh = i / d;
    const int c = (int)(i % d);
    const T* src = Qh + bh * n_hist * d + c;
    double acc = 0.0;
    for (int t = 0; t < n_hist; ++t) {
        const double q = load_f32(src + (long long)t * d);
        acc += q * q;
    }
    w[i] = (float)(acc / (double)n_hist);
}

// Residual variance of codebook keys, v_c = (1/n) sum_t (x_t - mu_a(t))^2, with the
// cache's fp32 centroids and the nearest index a(t) (fp64 distance, ties to the lower
// index, as the append stores it), summed in fp64; one CTA per (channel, kv head, batch).
template <typename T>
__global__ void __launch_bounds__(kCbThreads)
residual_var_kernel(const T* __restrict__ K, int n, int d, int Hkv, const float* __restrict__ cent,
                    float* __restrict__ var) {
    __shared__ double s_acc[kCbThreads / 32];
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const long long bh = (long long)b * Hkv + h;
    const float4 m4 = *reinterpret_cast<const float4*>(cent + (bh * d + c) * 4);
    const double mu[4] = {m4.x, m4.y, m4.z, m4.w};
    const T* src = K + bh * n * d + c;
    double acc = 0.0;
    for (int t = tid; t < n; t += kCbThreads) {
        const double x = load_f32(src + (long long)t * d);
        int k = 0;
        double best = fabs(x - mu[0]);
#pragma unroll
        for (int q = 1; q < 4; ++q) {
            const double dq = fabs(x - mu[q]);
            if (dq < best) {
                best = dq;
                k = q;
            }
        }
        const double e = x - mu[k];
        acc += e * e;
    }
    acc = warp_sum_d(acc);
    if ((tid & 31) == 0) s_acc[tid >> 5] = acc;
    __syncthreads();
    if (tid == 0) {
        double a = 0.0;
        for (int q = 0; q < kCbThreads / 32; ++q) a += s_acc[q];
        var[bh * d + c] = (float)(a / (double)n);
    }
}

// C = (1/n) sum_t q_t q_t^T in fp64, one CTA per (b, h); C [d][d] into the workspace.
template <typename T>
__global__ void __launch_bounds__(kJThreads)
second_moment_kernel(const T* __restrict__ Qh, int n_hist, int d, double* __restrict__ Cws) {
    const int bh = blockIdx.x;
    const T* src = Qh + (long long)bh * n_hist * d;
    double* C = Cws + (long long)bh * d * d;
    for (int e = threadIdx.x; e < d * d; e += kJThreads) {
        const int i = e / d, j = e % d;
        double acc = 0.0;
        for (int t = 0; t < n_hist; ++t) acc += (double)load_f32(src + (long long)t * d + i) * (double)load_f32(src + (long long)t * d + j);
        C[e] = acc / (double)n_hist;
    }
}

// Round-robin pairing of round `r` over indices 0..m-1 (m even): slot 0 fixed,
// the other m - 1 indices rotate; pair i joins positions i and m - 1 - i.
__device__ __forceinline__ int rr_index(int pos, int r, int m) { return pos == 0 ? 0 : 1 + (pos - 1 + r) % (m - 1); }

// Cyclic Jacobi eigen-decomposition of the symmetric C (fp64) of one (b, h), then
// the top-r eigenvectors, sign-fixed, as fp32 U [d][r] and the eigenvalues.
__global__ void __launch_bounds__(kJThreads)
jacobi_kernel(double* __restrict__ Cws, double* __restrict__ Vws, int d, int r, float* __restrict__ U,
              float* __restrict__ eig_out) {
    extern __shared__ double A[];               // [d][d]
    __shared__ double s_c[128], s_s[128];
    __shared__ int s_p[128], s_q[128];
    __shared__ double s_red[kJThreads / 32];
    __shared__ int s_order[256];
    __shared__ double s_done;
    const int bh = blockIdx.x, tid = threadIdx.x;
    double* V = Vws + (long long)bh * d * d;
    const double* C = Cws + (long long)bh * d * d;
    for (int e = tid; e < d * d; e += kJThreads) {
        A[e] = C[e];
        V[e] = (e / d == e % d) ? 1.0 : 0.0;
    }
    __syncthreads();
    const int m = d, half = d / 2;
    for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
        // convergence: off-diagonal mass against the diagonal
        double off = 0.0, dia = 0.0;
        for (int e = tid; e < d * d; e += kJThreads) {
            const double a = A[e];
            if (e / d == e % d) dia += a * a;
            else off += a * a;
        }
        off = warp_sum_d(off);
        dia = warp_sum_d(dia);
        if ((tid & 31) == 0) s_red[tid >> 5] = off;
        __syncthreads();
        if (tid == 0) {
            double o = 0.0;
            for (int w = 0; w < kJThreads / 32; ++w) o += s_red[w];
            s_done = o;
        }
        __syncthreads();
        const double offsum = s_done;
        __syncthreads();
        if ((tid & 31) == 0) s_red[tid >> 5] = dia;
        __syncthreads();
        if (tid == 0) {
            double o = 0.0;
            for (int w = 0; w < kJThreads / 32; ++w) o += s_red[w];
            s_done = o;
        }
        __syncthreads();
        if (offsum <= 1e-30 * s_done || offsum == 0.0) break;
        __syncthreads();
        for (int rd = 0; rd < m - 1; ++rd) {
            // rotation angles of this sweep step's d/2 disjoint pairs
            for (int i = tid; i < half; i += kJThreads) {
                int p = rr_index(i, rd, m), q = rr_index(m - 1 - i, rd, m);
                if (p > q) { const int t = p; p = q; q = t; }
                const double apq = A[p * d + q];
                double c = 1.0, s = 0.0;
                if (apq != 0.0) {
                    const double th = (A[q * d + q] - A[p * d + p]) / (2.0 * apq);
                    const double t = (th >= 0.0 ? 1.0 : -1.0) / (fabs(th) + sqrt(1.0 + th * th));
                    c = 1.0 / sqrt(1.0 + t * t);
                    s = t * c;
                }
                s_p[i] = p;
                s_q[i] = q;
                s_c[i] = c;
                s_s[i] = s;
            }
            __syncthreads();
            // rows: A <- J^T A
            for (int e = tid; e < half * d; e += kJThreads) {
                const int i = e / d, k = e % d;
                const int p = s_p[i], q = s_q[i];
                const double c = s_c[i], s = s_s[i];
                const double ap = A[p * d + k], aq = A[q * d + k];
                A[p * d + k] = c * ap - s * aq;
                A[q * d + k] = s * ap + c * aq;
            }
            __syncthreads();
            // columns: A <- A J, and V <- V J
            for (int e = tid; e < half * d; e += kJThreads) {
                const int i = e / d, k = e % d;
                const int p = s_p[i], q = s_q[i];
                const double c = s_c[i], s = s_s[i];
                const double ap = A[k * d + p], aq = A[k * d + q];
                A[k * d + p] = c * ap - s * aq;
                A[k * d + q] = s * ap + c * aq;
                const double vp = V[k * d + p], vq = V[k * d + q];
                V[k * d + p] = c * vp - s * vq;
                V[k * d + q] = s * vp + c * vq;
            }
            __syncthreads();
        }
    }
    // order of the eigenvalues, descending, ties to the lower index (rank counting)
    for (int i = tid; i < d; i += kJThreads) {
        const double li = A[i * d + i];
        int rank = 0;
        for (int j = 0; j < d; ++j) {
            const double lj = A[j * d + j];
            if (lj > li || (lj == li && j < i)) ++rank;
        }
        s_order[rank] = i;
    }
    __syncthreads();
    // top-r columns, each signed so that its largest-magnitude entry is positive
    for (int jr = tid; jr < r; jr += kJThreads) {
        const int col = s_order[jr];
        int arg = 0;
        double best = -1.0;
        for (int k = 0; k < d; ++k) {
            const double a = fabs(V[k * d + col]);
            if (a > best) {
                best = a;
                arg = k;
            }
        }
        const double sg = V[arg * d + col] < 0.0 ? -1.0 : 1.0;
        for (int k = 0; k < d; ++k) U[((long long)bh * d + k) * r + jr] = (float)(sg * V[k * d + col]);
        if (eig_out) eig_out[(long long)bh * r + jr] = (float)A[col * d + col];
    }
}

int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

size_t codebook_ws_bytes(const kv_layout* L, int n_tokens) {
    (void)L;
    (void)n_tokens;
    return 0;
}

kv_status launch_codebook_fit(const void* K, kv_dtype dt, int n_tokens, const kv_cache* cache, int iters,
                              const void* Qhist, int n_hist, float* weights_out, int range, void* ws, cudaStream_t st) {
    (void)ws;
    const kv_layout& L = cache->layout;
    if (n_tokens > kMaxCbTokens)
        return set_error(KV_ERR_UNSUPPORTED, "codebook fit: at most %d tokens per channel (got %d)", kMaxCbTokens,
                         n_tokens);
    const int npow2 = pow2_at_least(n_tokens);
    const size_t smem = (size_t)npow2 * sizeof(float);
    dim3 grid(L.d, L.Hkv, L.B);
    // the weights come first: the residual-range update reads them
#define BITKV_CB(T)                                                                                          \
    do {                                                                                                     \
        if (Qhist) {                                                                                         \
            const long long total = (long long)L.B * L.Hkv * L.d;                                            \
            sensitivity_kernel<T><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(static_cast<const T*>(Qhist), \
                                                                                  n_hist, L.d, total,        \
                                                                                  weights_out);              \
        }                                                                                                    \
        cudaFuncSetAttribute(codebook_fit_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        codebook_fit_kernel<T><<<grid, kCbThreads, smem, st>>>(static_cast<const T*>(K), n_tokens, npow2, L.d, \
                                                               L.Hkv, iters, range ? weights_out : nullptr, \
                                                               cache->centroids);                           \
    } while (0)
    switch (dt) {
        case KV_F32: BITKV_CB(float); break;
        case KV_F16: BITKV_CB(__half); break;
        case KV_BF16: BITKV_CB(__nv_bfloat16); break;
    }
#undef BITKV_CB
    return check_launch("codebook_fit_kernel");
}

kv_status launch_residual_var(const void* K, kv_dtype dt, int n_tokens, const kv_cache* cache, cudaStream_t st) {
    const kv_layout& L = cache->layout;
    dim3 grid(L.d, L.Hkv, L.B);
    switch (dt) {
        case KV_F32:
            residual_var_kernel<float><<<grid, kCbThreads, 0, st>>>(static_cast<const float*>(K), n_tokens, L.d, L.Hkv,
                                                                   cache->centroids, cache->resid_var);
            break;
        case KV_F16:
            residual_var_kernel<__half><<<grid, kCbThreads, 0, st>>>(static_cast<const __half*>(K), n_tokens, L.d,
                                                                    L.Hkv, cache->centroids, cache->resid_var);
            break;
        case KV_BF16:
            residual_var_kernel<__nv_bfloat16><<<grid, kCbThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(K),
                                                                           n_tokens, L.d, L.Hkv, cache->centroids,
                                                                           cache->resid_var);
            break;
    }
    return check_launch("residual_var_kernel");
}

size_t psac_ws_bytes(const kv_layout* L) {
    return (size_t)2 * L->B * L->Hkv * L->d * L->d * sizeof(double);
}

kv_status launch_psac_basis(const void* Qhist, kv_dtype dt, int n_hist, const kv_cache* cache, float* eig_out,
                            void* ws, cudaStream_t st) {
    const kv_layout& L = cache->layout;
    if (L.d > 128 || L.d % 2 != 0) return set_error(KV_ERR_UNSUPPORTED, "PSAC basis: d=%d must be even and <= 128", L.d);
    double* Cws = static_cast<double*>(ws);
    double* Vws = Cws + (size_t)L.B * L.Hkv * L.d * L.d;
    const int nbh = L.B * L.Hkv;
    switch (dt) {
        case KV_F32:
            second_moment_kernel<float><<<nbh, kJThreads, 0, st>>>(static_cast<const float*>(Qhist), n_hist, L.d, Cws);
            break;
        case KV_F16:
            second_moment_kernel<__half><<<nbh, kJThreads, 0, st>>>(static_cast<const __half*>(Qhist), n_hist, L.d, Cws);
            break;
        case KV_BF16:
            second_moment_kernel<__nv_bfloat16><<<nbh, kJThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(Qhist),
                                                                          n_hist, L.d, Cws);
            break;
    }
    kv_status s = check_launch("second_moment_kernel");
    if (s != KV_OK) return s;
    const size_t smem = (size_t)L.d * L.d * sizeof(double);
    cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    jacobi_kernel<<<nbh, kJThreads, smem, st>>>(Cws, Vws, L.d, L.psac_rank, cache->psac_u, eig_out);
    return check_launch("jacobi_kernel");
}

}  // namespace bitkv
