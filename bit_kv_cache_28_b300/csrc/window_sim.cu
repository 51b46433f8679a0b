// kv_window_similarity: the cosine similarity of every 32-token window of a key
// sequence to a question, the score that kv_window_plan ranks windows by
// (WindowQuant note, section 何が新しいのか: each window's similarity to the text
// question, by cosine similarity, picks its bit-width; 実装者視点で気になった点:
// windows of 32 tokens).
//
// A window is the mean of its valid tokens' keys and the question the mean of its
// tokens' keys, every kv head's d channels concatenated; the similarity is
// u.v / (|u| |v|), 0 where either vector is zero.  Cosine does not see the scale,
// so the kernel works with sums instead of means.
//
// Layout and roofline: K is read once, 16 bytes per thread per token, so the
// kernel is bound by HBM at B Hkv n d sizeof(T) bytes (plus the question, read
// once per CTA from L2).  Thread t of a window's team owns 16 bytes of channels
// of one kv head (h = t / (d / VEC)).  When a window's channels fit one warp
// (Hkv d sizeof(T) <= 512 bytes), each warp of a 4-warp CTA is a team of its
// own and the CTA's first warp sums the question once for all four; otherwise
// the whole CTA is one team and serves a few windows in turn.
#include <cmath>

#include "common.cuh"

namespace bitkv {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kWin = 32;            // tokens per window
constexpr int kWinPerCta = 4;       // windows one CTA serves (question sums amortised)

template <typename T> struct Vec;   // 16 bytes of T as floats
template <> struct Vec<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void add(float (&a)[4], const uint4& w) {
        a[0] += __uint_as_float(w.x); a[1] += __uint_as_float(w.y);
        a[2] += __uint_as_float(w.z); a[3] += __uint_as_float(w.w);
    }
};
template <> struct Vec<__half> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void add(float (&a)[8], const uint4& w) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[k]));
            a[2 * k] += f.x;
            a[2 * k + 1] += f.y;
        }
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void add(float (&a)[8], const uint4& w) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            a[2 * k] += __uint_as_float(u[k] << 16);
            a[2 * k + 1] += __uint_as_float(u[k] & 0xFFFF0000u);
        }
    }
};

// Adds a full window's 32 token rows (16 bytes each, `stride` uint4 apart) into u:
// 16 loads are issued before the first is used, so a warp keeps 8 KB in flight.
template <typename V>
__device__ __forceinline__ void add_window(float (&u)[V::N], const uint4* p, int stride) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint4 buf[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) buf[j] = __ldg(p + (long long)(16 * half + j) * stride);
#pragma unroll
        for (int j = 0; j < 16; ++j) V::add(u, buf[j]);
    }
}

// Sums two values over the CTA; every thread gets the totals.  red holds 2 floats
// per warp.
__device__ __forceinline__ float2 cta_sum2(float a, float b, float2* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if (nw == 1) return make_float2(a, b);
    __syncthreads();                                  // red is free (previous use read)
    if ((threadIdx.x & 31) == 0) red[warp] = make_float2(a, b);
    __syncthreads();
    float2 s = make_float2(0.0f, 0.0f);
    for (int w = 0; w < nw; ++w) {
        s.x += red[w].x;
        s.y += red[w].y;
    }
    return s;
}

template <typename T>
__global__ void __launch_bounds__(1024)
window_sim_kernel(const T* __restrict__ K, const T* __restrict__ Kq, int Hkv, int n, int m, int d, int W,
                  float* __restrict__ sim) {
    using V = Vec<T>;
    __shared__ float2 red[32];
    const int b = blockIdx.y;
    const int per_head = d / V::N, P = Hkv * per_head;
    const int t = threadIdx.x;
    const bool own = t < P;
    const int h = own ? t / per_head : 0, cg = own ? t - h * per_head : 0;
    // question sums of this thread's channels, and |v|^2
    float v[V::N];
#pragma unroll
    for (int k = 0; k < V::N; ++k) v[k] = 0.0f;
    if (own) {
        const uint4* q = reinterpret_cast<const uint4*>(Kq + ((long long)b * Hkv + h) * m * d) + cg;
        for (int j = 0; j < m; ++j) V::add(v, __ldg(q + (long long)j * per_head));
    }
    float vv = 0.0f;
#pragma unroll
    for (int k = 0; k < V::N; ++k) vv = fmaf(v[k], v[k], vv);
    vv = cta_sum2(vv, 0.0f, red).x;

    const uint4* kb = reinterpret_cast<const uint4*>(K + ((long long)b * Hkv + h) * n * d) + cg;
    for (int w = blockIdx.x; w < W; w += gridDim.x) {
        const int t0 = w * kWin, nt = min(kWin, n - t0);
        float u[V::N];
#pragma unroll
        for (int k = 0; k < V::N; ++k) u[k] = 0.0f;
        if (own) {
            const uint4* p = kb + (long long)t0 * per_head;
            if (nt == kWin) {
                add_window<V>(u, p, per_head);
            } else {
                for (int j = 0; j < nt; ++j) V::add(u, __ldg(p + (long long)j * per_head));
            }
        }
        float uv = 0.0f, uu = 0.0f;
#pragma unroll
        for (int k = 0; k < V::N; ++k) {
            uv = fmaf(u[k], v[k], uv);
            uu = fmaf(u[k], u[k], uu);
        }
        const float2 s = cta_sum2(uv, uu, red);
        if (t == 0) sim[(long long)b * W + w] = s.y > 0.0f && vv > 0.0f ? s.x / (sqrtf(s.y) * sqrtf(vv)) : 0.0f;
    }
}

// One warp per window (Hkv d / VEC <= 32 lanes), 4 windows per CTA: small CTAs let
// the whole grid of the decode workload's 4904 windows be resident in one wave
// (8-warp CTAs left a second, nearly empty wave; several windows per warp in turn
// expose the load latency of each).
constexpr int kTeams = 4;

template <typename T>
__global__ void __launch_bounds__(32 * kTeams)
window_sim_warp_kernel(const T* __restrict__ K, const T* __restrict__ Kq, int Hkv, int n, int m, int d, int W,
                       float* __restrict__ sim) {
    using V = Vec<T>;
    __shared__ float vsh[V::N][32];
    __shared__ float vv_sh;
    const int b = blockIdx.y, lane = threadIdx.x & 31, team = threadIdx.x >> 5;
    const int per_head = d / V::N, P = Hkv * per_head;
    const bool own = lane < P;
    const int h = own ? lane / per_head : 0, cg = own ? lane - h * per_head : 0;
    if (team == 0) {
        float v[V::N];
#pragma unroll
        for (int k = 0; k < V::N; ++k) v[k] = 0.0f;
        if (own) {
            const uint4* q = reinterpret_cast<const uint4*>(Kq + ((long long)b * Hkv + h) * m * d) + cg;
            for (int j = 0; j < m; ++j) V::add(v, __ldg(q + (long long)j * per_head));
        }
        float vv = 0.0f;
#pragma unroll
        for (int k = 0; k < V::N; ++k) {
            vv = fmaf(v[k], v[k], vv);
            vsh[k][lane] = v[k];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) vv += __shfl_xor_sync(0xffffffffu, vv, o);
        if (lane == 0) vv_sh = vv;
    }
    __syncthreads();
    float v[V::N];
#pragma unroll
    for (int k = 0; k < V::N; ++k) v[k] = vsh[k][lane];
    const float vv = vv_sh;
    const uint4* kb = reinterpret_cast<const uint4*>(K + ((long long)b * Hkv + h) * n * d) + cg;
    for (int w = blockIdx.x * kTeams + team; w < W; w += gridDim.x * kTeams) {
        const int t0 = w * kWin, nt = min(kWin, n - t0);
        float u[V::N];
#pragma unroll
        for (int k = 0; k < V::N; ++k) u[k] = 0.0f;
        if (own) {
            const uint4* p = kb + (long long)t0 * per_head;
            if (nt == kWin) {
                add_window<V>(u, p, per_head);
            } else {
                for (int j = 0; j < nt; ++j) V::add(u, __ldg(p + (long long)j * per_head));
            }
        }
        float uv = 0.0f, uu = 0.0f;
#pragma unroll
        for (int k = 0; k < V::N; ++k) {
            uv = fmaf(u[k], v[k], uv);
            uu = fmaf(u[k], u[k], uu);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            uv += __shfl_xor_sync(0xffffffffu, uv, o);
            uu += __shfl_xor_sync(0xffffffffu, uu, o);
        }
        if (lane == 0) sim[(long long)b * W + w] = uu > 0.0f && vv > 0.0f ? uv / (sqrtf(uu) * sqrtf(vv)) : 0.0f;
    }
}

template <typename T>
kv_status launch_window_sim(const void* K, const void* Kq, int B, int Hkv, int n, int m, int d, float* sim,
                            cudaStream_t st) {
    const int W = (n + kWin - 1) / kWin;
    const int P = Hkv * (d / Vec<T>::N);
    if (P <= 32) {
        dim3 grid((W + kTeams - 1) / kTeams, B);
        window_sim_warp_kernel<T><<<grid, 32 * kTeams, 0, st>>>(static_cast<const T*>(K), static_cast<const T*>(Kq),
                                                                Hkv, n, m, d, W, sim);
        return check_launch("window_sim_warp_kernel");
    }
    const int threads = (P + 31) / 32 * 32;
    dim3 grid((W + kWinPerCta - 1) / kWinPerCta, B);
    window_sim_kernel<T><<<grid, threads, 0, st>>>(static_cast<const T*>(K), static_cast<const T*>(Kq), Hkv, n, m, d,
                                                   W, sim);
    return check_launch("window_sim_kernel");
}

}  // namespace
}  // namespace bitkv

using namespace bitkv;

extern "C" kv_status kv_window_similarity(const void* K, const void* Kq, kv_dtype dtype, int B, int Hkv, int n, int m,
                                          int d, float* sim, void* stream) {
    AbiRange nvtx_range("kv_window_similarity");
    if (B <= 0 || Hkv <= 0 || d <= 0 || n < 0 || m < 0)
        return set_error(KV_ERR_INVALID_ARG, "kv_window_similarity: bad sizes B=%d Hkv=%d n=%d m=%d d=%d", B, Hkv, n,
                         m, d);
    if (dtype < KV_F32 || dtype > KV_BF16) return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (n == 0) return KV_OK;
    if (!K || !sim || (m > 0 && !Kq)) return set_error(KV_ERR_INVALID_ARG, "kv_window_similarity: NULL pointer");
    const int esize = dtype == KV_F32 ? 4 : 2;
    if ((d * esize) % 16 != 0)
        return set_error(KV_ERR_UNSUPPORTED, "kv_window_similarity: rows of d=%d must be a multiple of 16 bytes", d);
    if (Hkv * d * esize / 16 > 1024)
        return set_error(KV_ERR_UNSUPPORTED, "kv_window_similarity: Hkv*d=%d channels exceed one CTA", Hkv * d);
    if (B > 65535) return set_error(KV_ERR_UNSUPPORTED, "kv_window_similarity: B=%d above 65535", B);
    if (!aligned16(K) || (m > 0 && !aligned16(Kq)) || (reinterpret_cast<uintptr_t>(sim) & 3u))
        return set_error(KV_ERR_ALIGNMENT, "kv_window_similarity: K and Kq must be 16-byte aligned, sim 4-byte");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
        case KV_F32: return launch_window_sim<float>(K, Kq, B, Hkv, n, m, d, sim, st);
        case KV_F16: return launch_window_sim<__half>(K, Kq, B, Hkv, n, m, d, sim, st);
        default: return launch_window_sim<__nv_bfloat16>(K, Kq, B, Hkv, n, m, d, sim, st);
    }
}
