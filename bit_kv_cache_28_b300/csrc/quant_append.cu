// kv_quantize_append kernels: quantise one finished chunk (or one prefill of
// windows) and pack it into the cache's blocks, plus the debug dequantiser.
//
// "Quantized Keys Steal Attention" (abstract): the cache of previously
// generated chunks is stored at INT2 with per-key step sizes.  WindowQuant
// note (技術的に面白い点, 実装者視点で気になった点): 32-token windows with one
// bit-width each, stored grouped by bit-width.  "QuantWM" (Innovations 2, 3):
// codebook key indices plus PSAC coefficients.
//
// One CTA packs one 32-token block of one (batch, kv head): the block's key
// and value rows are staged in shared memory as fp32; each key channel and each
// (token, 32-channel value group) is reduced by 256/d adjacent threads with
// shuffle min/max, the codes go to byte scratch arrays, and one thread per
// output word packs them.
#include <cstdio>

#include "common.cuh"

namespace bitkv {

namespace {

constexpr int kAppendThreads = 256;

// 16 bytes of the input dtype as fp32 values (8 for 16-bit types, 4 for fp32).
template <typename T> __device__ __forceinline__ void widen16(uint4 v, float* out);
template <> __device__ __forceinline__ void widen16<float>(uint4 v, float* out) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void widen16<__nv_bfloat16>(uint4 v, float* out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        out[2 * k] = __uint_as_float(w[k] << 16);
        out[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
template <> __device__ __forceinline__ void widen16<__half>(uint4 v, float* out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        out[2 * k] = f.x;
        out[2 * k + 1] = f.y;
    }
}

__device__ __forceinline__ void step_and_zero(float mn, float mx, float qmax, float& s, float& z) {
    z = __fadd_rn(mn, 0.0f);                         // -0.0 -> +0.0
    s = __fadd_rn(__fdiv_rn(__fsub_rn(mx, z), qmax), 0.0f);
}

// The stored (s, z) of a group: the fp32 pair, or its fp16 rounding (RNE; a -0 zero
// point becomes +0) whose exact widening then serves for the codes.
__device__ __forceinline__ void store_meta(unsigned char* base, int i, int meta16, float& s, float& z, bool write) {
    if (meta16) {
        const __half2 h = __floats2half2_rn(s, __fadd_rn(__half2float(__float2half_rn(z)), 0.0f));
        const float2 f = __half22float2(h);
        s = f.x;
        z = f.y;
        if (write) reinterpret_cast<__half2*>(base)[i] = h;
    } else if (write) {
        reinterpret_cast<float2*>(base)[i] = make_float2(s, z);
    }
}

// Code of d = fl32(x - z) for step s with inverse r = 1/s (rounded): rint(fl32(d / s)),
// clamped.  fl32(d * r) lies within 3 * 2^-24 |d / s| of fl32(d / s) (both quotients
// carry at most two roundings of 2^-24), so the two round to the same integer
// unless one sits within 4e-6 of a half-integer; there the IEEE division decides.
__device__ __forceinline__ uint32_t code_fast(float x, float s, float r, float z, float qmax) {
    if (!(s > 0.0f)) return 0u;
    const float d = __fsub_rn(x, z);
    float q = __fmul_rn(d, r);
    const float fr = q - floorf(q);
    if (fabsf(fr - 0.5f) < 4e-6f || !(r < INFINITY)) q = __fdiv_rn(d, s);
    return static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.0f), qmax));
}

// Values of one block, INT layout: (token t, 32-channel group g) is shared by
// tpc = 256 / d adjacent threads, each taking 32 / tpc channels; min / max are
// combined by shuffles.  Writes Vm[g][t] (fp32 or fp16 pairs) and the codes into vc8[c][t].
template <int BITS>
__device__ void encode_values(const float* Vs, int ld, int d, int nv, uint8_t* vc8, unsigned char* vm, int meta16) {
    const float qmax = float((1 << BITS) - 1);
    const int tid = threadIdx.x;
    const int tpc = kAppendThreads / d, span = kBlockTokens / tpc, part = tid % tpc;
    const int ng = d / 32, pr = tid / tpc;
    const int t = pr / ng, g = pr % ng, c0 = g * 32 + part * span;
    float mn = INFINITY, mx = -INFINITY;
    if (t < nv)
        for (int i = 0; i < span; ++i) {
            const float x = Vs[t * ld + c0 + i];
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
    for (int w = 1; w < tpc; w <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, w));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
    }
    float s = 0.0f, z = 0.0f;
    if (t < nv) step_and_zero(mn, mx, qmax, s, z);
    store_meta(vm, g * 32 + t, meta16, s, z, part == 0);
    const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
    for (int i = 0; i < span; ++i)
        vc8[(c0 + i) * kBlockTokens + t] =
            t < nv ? static_cast<uint8_t>(code_fast(Vs[t * ld + c0 + i], s, r, z, qmax)) : 0;
}

// Pack byte codes into b-bit words: word w holds bytes w per .. w per + per - 1
// (per = 32 / b), byte i at bits [b i, b i + b).  The key bytes are token-major
// and the value bytes channel-major, so the same rule gives both layouts.
template <int BITS>
__device__ void pack_words(const uint8_t* kc8, const uint8_t* vc8, int nwords, uint32_t* kw, uint32_t* vw) {
    constexpr int per = 32 / BITS;
    for (int w = threadIdx.x; w < nwords; w += kAppendThreads) {
        const uint8_t* ksrc = kc8 + w * per;
        const uint8_t* vsrc = vc8 + w * per;
        uint32_t a = 0, bq = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) {
            a |= uint32_t(ksrc[i]) << (BITS * i);
            bq |= uint32_t(vsrc[i]) << (BITS * i);
        }
        kw[w] = a;
        vw[w] = bq;
    }
}

// One uniform INT block.  Keys: channel c is shared by tpc = 256 / d adjacent
// threads, each taking 32 / tpc tokens; min / max are combined by shuffles.
// Values as encode_values.  Codes go to byte arrays kc8[t][c] and vc8[c][t];
// one thread per output word packs them.
template <int BITS>
__device__ void encode_int_block(const float* Ks, const float* Vs, int ld, int d, int nv, uint8_t* kc8,
                                 uint8_t* vc8, unsigned char* blk, int meta16) {
    const float qmax = float((1 << BITS) - 1);
    const IntBlockOffsets o = int_offsets(d, BITS, meta16);
    const int tid = threadIdx.x;
    const int tpc = kAppendThreads / d;           // 1, 2, 4 or 8 threads per group
    const int span = kBlockTokens / tpc;          // elements per thread
    const int part = tid % tpc;
    // keys: per channel over the block's valid tokens
    {
        const int ch = tid / tpc, t0 = part * span;
        float mn = INFINITY, mx = -INFINITY;
        for (int i = 0; i < span; ++i) {
            const int t = t0 + i;
            if (t < nv) {
                const float x = Ks[t * ld + ch];
                mn = fminf(mn, x);
                mx = fmaxf(mx, x);
            }
        }
        for (int w = 1; w < tpc; w <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, w));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, w));
        }
        float s = 0.0f, z = 0.0f;
        if (nv > 0) step_and_zero(mn, mx, qmax, s, z);
        store_meta(blk + o.km, ch, meta16, s, z, part == 0);
        const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
        for (int i = 0; i < span; ++i) {
            const int t = t0 + i;
            kc8[t * d + ch] = t < nv ? static_cast<uint8_t>(code_fast(Ks[t * ld + ch], s, r, z, qmax)) : 0;
        }
    }
    encode_values<BITS>(Vs, ld, d, nv, vc8, blk + o.vm, meta16);
    __syncthreads();
    pack_words<BITS>(kc8, vc8, kBlockTokens * d * BITS / 32, reinterpret_cast<uint32_t*>(blk + o.kc),
                     reinterpret_cast<uint32_t*>(blk + o.vc));
}

// Exact sum s + e = a + b of two floats (Knuth's TwoSum; no FMA contraction).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Packed fp32 pairs (sm_100+ f32x2 instructions: one instruction, two lanes of work).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 x2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 x2_split(f32x2 v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f32x2 x2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 x2_sub(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 x2_mul(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 x2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// One compensated dot-product step for two ranks: (s, cc) += u (eh + el), with the
// product u eh split exactly by FMA and the sum split exactly by TwoSum.
__device__ __forceinline__ void dot2_step(f32x2& s, f32x2& cc, f32x2 u, f32x2 eh, f32x2 el) {
    const f32x2 p = x2_mul(u, eh);
    const f32x2 pe = x2_fma(u, el, x2_fma(u, eh, p ^ 0x8000000080000000ull));
    const f32x2 s2 = x2_add(s, p);
    const f32x2 bp = x2_sub(s2, s);
    const f32x2 err = x2_add(x2_sub(s, x2_sub(s2, bp)), x2_sub(p, bp));
    s = s2;
    cc = x2_add(cc, x2_add(err, pe));
}
// (s, cc) += (s', cc') for two ranks, the high parts added exactly by TwoSum.
__device__ __forceinline__ void dot2_merge(f32x2& s, f32x2& cc, f32x2 so, f32x2 co) {
    const f32x2 s2 = x2_add(s, so);
    const f32x2 bp = x2_sub(s2, s);
    const f32x2 err = x2_add(x2_sub(s, x2_sub(s2, bp)), x2_sub(so, bp));
    s = s2;
    cc = x2_add(x2_add(cc, co), err);
}

// Nearest-centroid rule of one channel as fp32 comparisons.  The centroids
// sorted ascending by (value, index), v_0 <= .. <= v_3, each position carrying
// the lowest index that holds its value (rep), split the line at the midpoints
// M_i = (v_i + v_{i+1}) / 2: x is nearest to v_c with c = #{i : x > M_i}, and
// x == M_c is a tie between v_c and v_{c+1} that goes to the lower index (equal
// neighbours share rep, so their midpoint changes nothing).  For an fp32 x,
// x > M exactly when x > RD32(M), and x == M only if M is an fp32 value; M comes
// exactly from the TwoSum a + b = s + e as s / 2 + e / 2 (RD32(M) = s / 2 if
// e >= 0, else the float below it; an fp32 value iff e == 0).  Centroids must be
// finite, with pairwise sums of magnitude >= 2^-125 or zero (s / 2 exact).
//
// The rule is the exact nearest centroid; fp64 |x - mu| is exact too unless x and
// a nonzero mu differ by more than 2^29 in magnitude.  There (|x| below 2^-28 of
// the largest |mu| or above 2^28 of the smallest nonzero |mu|) the fp64 distances
// are compared directly, first minimum winning, so that both agree everywhere.
struct CentroidRule {
    float thr[3];     // RD32(M_i)
    float teq[3];     // M_i when it is an fp32 value, else NaN
    uint32_t rep;     // byte c: index of v_c (lowest index of its value)
    uint32_t tie;     // byte c: min(rep_c, rep_{c+1})
    float tiny, huge; // |x| < tiny or |x| > huge: fp64 comparison
};

__device__ __forceinline__ CentroidRule centroid_rule(float4 mu) {
    float v[4] = {mu.x, mu.y, mu.z, mu.w};
    int id[4] = {0, 1, 2, 3};
    // sort (value, index) ascending: 5 compare-exchanges
    auto cx = [&](int i, int j) {
        if (v[i] > v[j] || (v[i] == v[j] && id[i] > id[j])) {
            const float tv = v[i];
            v[i] = v[j];
            v[j] = tv;
            const int ti = id[i];
            id[i] = id[j];
            id[j] = ti;
        }
    };
    cx(0, 1);
    cx(2, 3);
    cx(0, 2);
    cx(1, 3);
    cx(1, 2);
    int rp[4];
    rp[0] = id[0];
#pragma unroll
    for (int k = 1; k < 4; ++k) rp[k] = v[k] == v[k - 1] ? rp[k - 1] : id[k];
    CentroidRule R;
    float amax = 0.0f, amin = INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = fabsf(v[k]);
        amax = fmaxf(amax, a);
        if (a > 0.0f) amin = fminf(amin, a);
    }
    R.tiny = amax * 3.7252902984619141e-09f;     // 2^-28
    R.huge = amin * 268435456.0f;                // 2^28 (inf when every mu is 0)
    R.rep = (uint32_t)rp[0] | ((uint32_t)rp[1] << 8) | ((uint32_t)rp[2] << 16) | ((uint32_t)rp[3] << 24);
    R.tie = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        float s, e;
        two_sum(v[i], v[i + 1], s, e);
        const float h = __fmul_rn(s, 0.5f);
        // the float below h (h != 0 when e != 0: a nonzero exact sum never rounds to 0)
        const float below = __int_as_float(__float_as_int(h) + (h > 0.0f ? -1 : 1));
        R.thr[i] = e >= 0.0f ? h : below;
        R.teq[i] = e == 0.0f ? h : __int_as_float(0x7FC00000);
        R.tie |= (uint32_t)min(rp[i], rp[i + 1]) << (8 * i);
    }
    return R;
}

__device__ __noinline__ uint32_t nearest_centroid_f64(float4 mu, float x) {
    const double xd = x;
    const double d0 = fabs(xd - (double)mu.x), d1 = fabs(xd - (double)mu.y), d2 = fabs(xd - (double)mu.z),
                 d3 = fabs(xd - (double)mu.w);
    uint32_t k = 0;
    double best = d0;
    if (d1 < best) { best = d1; k = 1; }
    if (d2 < best) { best = d2; k = 2; }
    if (d3 < best) k = 3;
    return k;
}

__device__ __forceinline__ uint32_t nearest_centroid(const CentroidRule& R, float4 mu, float x) {
    const float ax = fabsf(x);
    if (!(ax < INFINITY)) return 0u;                 // NaN / inf: every distance ties -> index 0
    if (ax != 0.0f && (ax < R.tiny || ax > R.huge)) return nearest_centroid_f64(mu, x);
    const int c = (x > R.thr[0]) + (x > R.thr[1]) + (x > R.thr[2]);
    const float q = c == 0 ? R.teq[0] : (c == 1 ? R.teq[1] : R.teq[2]);
    const uint32_t w = (c < 3 && x == q) ? R.tie : R.rep;
    return (w >> (8 * c)) & 3u;
}

// Codebook block: the nearest fp32 centroid per key entry (ties to the lower
// index), INT2 values, fp16 PSAC coefficients U^T (k - k_hat).  The residual
// k - k_hat is kept exactly as a float pair and each coefficient is a
// compensated dot product (TwoProduct by FMA, TwoSum accumulation: the result
// of twice-fp32 precision), added in fp64 and rounded once to fp16.
__device__ void encode_cb_block(float* Ks, float* Vs, int ld, int d, int nv, uint8_t* kc8, uint8_t* vc8,
                                float* Us, unsigned char* blk, const float* cent, const float* U, int r, int rp) {
    const CbBlockOffsets o = cb_offsets(d);
    const int tid = threadIdx.x;
    for (int e = tid; e < d * rp; e += kAppendThreads) {
        const int c = e / rp, j = e - (e / rp) * rp;
        Us[e] = j < r ? __ldg(U + c * r + j) : 0.0f;
    }
    encode_values<2>(Vs, ld, d, nv, vc8, blk + o.vm, 0);
    __syncthreads();     // V is free for the low parts of the residual
    // keys: channel ch by tpc adjacent threads; the residual pair (high, low)
    // overwrites (K, V) in place
    const int tpc = kAppendThreads / d, span = kBlockTokens / tpc, part = tid % tpc;
    const int ch = tid / tpc, t0 = part * span;
    const float4 mu = __ldg(reinterpret_cast<const float4*>(cent) + ch);
    const CentroidRule R = centroid_rule(mu);
    for (int i = 0; i < span; ++i) {
        const int t = t0 + i;
        const float x = Ks[t * ld + ch];
        const uint32_t k = t < nv ? nearest_centroid(R, mu, x) : 0u;
        kc8[t * d + ch] = static_cast<uint8_t>(k);
        float eh = 0.0f, el = 0.0f;
        const float kh = k == 0 ? mu.x : (k == 1 ? mu.y : (k == 2 ? mu.z : mu.w));
        if (t < nv) two_sum(x, -kh, eh, el);
        Ks[t * ld + ch] = eh;
        Vs[t * ld + ch] = el;
    }
    __syncthreads();
    pack_words<2>(kc8, vc8, kBlockTokens * d / 16, reinterpret_cast<uint32_t*>(blk + o.kc),
                  reinterpret_cast<uint32_t*>(blk + o.vc));
    if (rp == 0) return;
    // coefficients: thread (token t, part) sums channels part, part + 8, .. for 8
    // ranks at a time from U staged as [d][rp] (zero past r); the 8 parts of a token
    // are adjacent lanes, merged by a TwoSum butterfly that leaves the same pair in
    // each of them
    const float4* Us4 = reinterpret_cast<const float4*>(Us);
    __half* kq = reinterpret_cast<__half*>(blk + o.kq);
    const int t = tid >> 3, prt = tid & 7;
    const float* ehr = Ks + t * ld;
    const float* elr = Vs + t * ld;
    for (int j0 = 0; j0 < rp; j0 += 8) {
        f32x2 sa[4], ca[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sa[k] = ca[k] = 0ull;
        if (t < nv) {
#pragma unroll 4
            for (int c = prt; c < d; c += 8) {
                const float eh = ehr[c], el = elr[c];
                const f32x2 eh2 = x2(eh, eh), el2 = x2(el, el);
                const float4 u0 = Us4[(c * rp + j0) >> 2], u1 = Us4[((c * rp + j0) >> 2) + 1];
                dot2_step(sa[0], ca[0], x2(u0.x, u0.y), eh2, el2);
                dot2_step(sa[1], ca[1], x2(u0.z, u0.w), eh2, el2);
                dot2_step(sa[2], ca[2], x2(u1.x, u1.y), eh2, el2);
                dot2_step(sa[3], ca[3], x2(u1.z, u1.w), eh2, el2);
            }
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dot2_merge(sa[k], ca[k], __shfl_xor_sync(0xffffffffu, sa[k], m),
                           __shfl_xor_sync(0xffffffffu, ca[k], m));
        // lane part writes rank j0 + part
        float sv = 0.0f, cv = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 a2 = x2_split(sa[k]), c2 = x2_split(ca[k]);
            if (prt == 2 * k) { sv = a2.x; cv = c2.x; }
            if (prt == 2 * k + 1) { sv = a2.y; cv = c2.y; }
        }
        const int j = j0 + prt;
        kq[t * rp + j] = (t < nv && j < r) ? __double2half((double)sv + (double)cv) : __float2half_rn(0.0f);
    }
}

// mode 0: uniform (segment `uni_seg`), 1: mixed (class per window), 2: codebook.
template <typename T>
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const T* __restrict__ K, const T* __restrict__ V, int n_tokens, DevCache c, int mode, int uni_seg,
              const int8_t* __restrict__ win_bits, int n_win, int tok0) {
    extern __shared__ float smem[];
    __shared__ int s_rank;
    const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int d = c.d, ld = d + 1;
    float* Ks = smem;
    float* Vs = Ks + kBlockTokens * ld;
    uint8_t* codes = reinterpret_cast<uint8_t*>(Vs + kBlockTokens * ld);
    const int t0 = j * kBlockTokens;
    const int nv = min(kBlockTokens, n_tokens - t0);

    int seg = uni_seg, idx;
    if (mode == 1) {
        const int bits = win_bits[(long long)b * n_win + j];
        seg = bits == 16 ? KV_SEG_RAW16 : (bits == 4 ? KV_SEG_INT4 : KV_SEG_INT2);
        if (threadIdx.x == 0) s_rank = 0;
        __syncthreads();
        int cnt = 0;
        for (int w = threadIdx.x; w < j; w += blockDim.x) cnt += win_bits[(long long)b * n_win + w] == bits;
        if (cnt) atomicAdd(&s_rank, cnt);
        __syncthreads();
        idx = c.n_blocks[seg] + s_rank;
    } else {
        idx = c.n_blocks[seg] + j;
    }
    unsigned char* blk = block_ptr(c, b, h, seg, idx);
    const long long row0 = (((long long)b * c.Hkv + h) * n_tokens + t0) * d;
    const int cls = seg_class(c.kind, seg);

    if (cls == CLS_RAW16) {
        // 16-bit windows keep the input bits unchanged (the dtype equals raw_dtype),
        // each row's 16-byte chunks moved to their permuted positions
        uint4* rk = reinterpret_cast<uint4*>(blk);
        const uint4* Kb = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(K) + row0);
        const uint4* Vb = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(V) + row0);
        const int nch = d / 8;
        for (int e = threadIdx.x; e < kBlockTokens * nch; e += blockDim.x) {
            const int t = e / nch, j = e % nch;
            const int dst = raw16_slot(t, 8 * j, d) >> 3;
            rk[dst] = t < nv ? Kb[e] : make_uint4(0, 0, 0, 0);
            rk[kBlockTokens * nch + dst] = t < nv ? Vb[e] : make_uint4(0, 0, 0, 0);
        }
    } else {
        // 16-byte vector loads of the block's rows, widened to fp32
        constexpr int VE = 16 / (int)sizeof(T);
        for (int e = threadIdx.x; e < kBlockTokens * d / VE; e += blockDim.x) {
            const int t = (e * VE) / d, ch = (e * VE) % d;
            float kf[VE], vf[VE];
            if (t < nv) {
                widen16<T>(*reinterpret_cast<const uint4*>(K + row0 + (long long)e * VE), kf);
                widen16<T>(*reinterpret_cast<const uint4*>(V + row0 + (long long)e * VE), vf);
            } else {
#pragma unroll
                for (int i = 0; i < VE; ++i) kf[i] = vf[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < VE; ++i) {
                Ks[t * ld + ch + i] = kf[i];
                Vs[t * ld + ch + i] = vf[i];
            }
        }
        __syncthreads();
        if (cls == CLS_INT4) {
            encode_int_block<4>(Ks, Vs, ld, d, nv, codes, codes + kBlockTokens * d, blk, c.meta16);
        } else if (cls == CLS_INT2) {
            encode_int_block<2>(Ks, Vs, ld, d, nv, codes, codes + kBlockTokens * d, blk, c.meta16);
        } else {
            const long long bh = (long long)b * c.Hkv + h;
            encode_cb_block(Ks, Vs, ld, d, nv, codes, codes + kBlockTokens * d,
                            reinterpret_cast<float*>(codes + 2 * kBlockTokens * d), blk, c.centroids + bh * d * 4,
                            c.r > 0 ? c.psac_u + bh * d * c.r : nullptr, c.r, c.rp);
        }
    }
    if (h == 0 && threadIdx.x == 0) {
        const long long gi = (long long)b * c.cap_total + c.seg_base[seg] + idx;
        c.blk_len[gi] = nv;
        c.blk_pos[gi] = tok0 + t0;
    }
}

// ---- uniform INT blocks from 16-bit rows, head dim 128: one CTA (8 warps) per block --------
// The same quantiser as encode_int_block with less work per element.
//   keys: the block's rows staged as raw 16-bit pairs in a 32 x 64-word tile whose 16-byte
//     chunks are XOR-swizzled by row / 8 (the reads below are then conflict-free); pad rows
//     hold a copy of row 0, so min / max over all 32 rows are those of the valid rows.  Warp w
//     owns channels 16 w .. 16 w + 15 (8 channel pairs), lane l the pair l / 4 over tokens
//     8 (l & 3) .. + 7: min / max by fp16x2 / bf16x2 operations (exact), two xor-shuffles, the
//     codes in registers, and each token's code word OR-reduced across the 8 (4) lanes that hold
//     its channels and stored directly (zero for pad tokens).
//   values: lane l of warp w takes token 4 w + l / 8, channels 16 (l & 7) .. + 15 straight from
//     global memory; a 32-channel group is two lanes (one shuffle); the codes go to a byte tile
//     [128 channels][32 tokens], from which each thread packs its channel-major words.
template <typename T> struct Pair16;
template <> struct Pair16<__half> {
    using P = __half2;
    static __device__ __forceinline__ float2 f2(uint32_t w) { return __half22float2(*reinterpret_cast<const P*>(&w)); }
    static __device__ __forceinline__ uint32_t mn(uint32_t a, uint32_t b) {
        const P r = __hmin2(*reinterpret_cast<const P*>(&a), *reinterpret_cast<const P*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    static __device__ __forceinline__ uint32_t mx(uint32_t a, uint32_t b) {
        const P r = __hmax2(*reinterpret_cast<const P*>(&a), *reinterpret_cast<const P*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
};
template <> struct Pair16<__nv_bfloat16> {
    using P = __nv_bfloat162;
    static __device__ __forceinline__ float2 f2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    static __device__ __forceinline__ uint32_t mn(uint32_t a, uint32_t b) {
        const P r = __hmin2(*reinterpret_cast<const P*>(&a), *reinterpret_cast<const P*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
    static __device__ __forceinline__ uint32_t mx(uint32_t a, uint32_t b) {
        const P r = __hmax2(*reinterpret_cast<const P*>(&a), *reinterpret_cast<const P*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
};

constexpr int kFastD = 128;

// Codes of two elements as code_fast() takes them (x0 against s0, r0 = 1/s0, z0; x1 against
// s1, r1, z1), in packed fp32x2 arithmetic: q = fl32(fl32(x - z) r) is rounded to the nearest
// integer, ties to even, by adding 1.5 2^23 (exact for |q| < 2^22, which a code's quotient
// always is) and read out of that sum's low mantissa bits.  e = q - rint(q) is exact, and
// ||e| - 1/2| equals code_fast()'s |q - floor(q) - 1/2| bit for bit, so the same elements (within
// 4e-6 of a half-integer, or r not finite) take the IEEE quotient.  With |e| <= 1/2 that test is
// one comparison: ||e| - 1/2| < 4e-6 (fp32) holds exactly when |e| > kTie, the float below
// 0.4999960065 (checked over every fp32 in [0, 1/2]).  A zero step comes with r = 0, so its q
// is 0 and its code 0.
__device__ __forceinline__ void code_pair2(float x0, float x1, float s0, float s1, float r0, float r1, float z0,
                                           float z1, int qmax, uint32_t& c0, uint32_t& c1) {
    constexpr float kMagic = 12582912.0f;   // 1.5 2^23
    const float kTie = __uint_as_float(0x3EFFFF79u);
    const f32x2 d = x2_sub(x2(x0, x1), x2(z0, z1));
    const f32x2 q = x2_mul(d, x2(r0, r1));
    const f32x2 t = x2_add(q, x2(kMagic, kMagic));
    const float2 e = x2_split(x2_sub(q, x2_sub(t, x2(kMagic, kMagic))));
    float2 tf = x2_split(t);
    if (fabsf(e.x) > kTie || !(r0 < INFINITY)) tf.x = __fadd_rn(__fdiv_rn(__fsub_rn(x0, z0), s0), kMagic);
    if (fabsf(e.y) > kTie || !(r1 < INFINITY)) tf.y = __fadd_rn(__fdiv_rn(__fsub_rn(x1, z1), s1), kMagic);
    const int k0 = (int)__float_as_uint(tf.x) - 0x4B400000, k1 = (int)__float_as_uint(tf.y) - 0x4B400000;
    c0 = (uint32_t)min(max(k0, 0), qmax);
    c1 = (uint32_t)min(max(k1, 0), qmax);
}

template <typename T, int BITS>
__global__ void __launch_bounds__(kAppendThreads)
append_int128_kernel(const T* __restrict__ K, const T* __restrict__ V, int n_tokens, DevCache c, int seg, int tok0) {
    using PP = Pair16<T>;
    constexpr int D = kFastD;
    constexpr float qmax = float((1 << BITS) - 1);
    __shared__ __align__(16) uint32_t kt[kBlockTokens * D / 2];     // 8 KB: key rows, 16-bit pairs
    __shared__ __align__(16) uint8_t vc8[D * kBlockTokens];         // 4 KB: value codes [c][t]
    const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = j * kBlockTokens;
    const int nv = min(kBlockTokens, n_tokens - t0);
    const int idx = c.n_blocks[seg] + j;
    unsigned char* blk = block_ptr(c, b, h, seg, idx);
    const IntBlockOffsets o = int_offsets(D, BITS, c.meta16);
    const long long row0 = (((long long)b * c.Hkv + h) * n_tokens + t0) * D;

    // key rows -> the swizzled tile (pad rows: a copy of row 0)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int e = tid + k * kAppendThreads, row = e >> 4, ch = e & 15;
        const int src = row < nv ? row : 0;
        const uint4 v = *reinterpret_cast<const uint4*>(K + row0 + (long long)src * D + 8 * ch);
        *reinterpret_cast<uint4*>(kt + row * (D / 2) + 4 * (ch ^ (((row >> 3) & 3) << 1))) = v;
    }

    // values: token tv, channels 16 jv .. 16 jv + 15 from global memory
    {
        const int tv = 4 * warp + (lane >> 3), jv = lane & 7;
        uint32_t w[8];
        if (tv < nv) {
            const uint4* src = reinterpret_cast<const uint4*>(V + row0 + (long long)tv * D + 16 * jv);
            const uint4 a = src[0], bq = src[1];
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = bq.x; w[5] = bq.y; w[6] = bq.z; w[7] = bq.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0u;
        }
        uint32_t mnp = w[0], mxp = w[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            mnp = PP::mn(mnp, w[i]);
            mxp = PP::mx(mxp, w[i]);
        }
        float2 fmn = PP::f2(mnp), fmx = PP::f2(mxp);
        float mn = fminf(fmn.x, fmn.y), mx = fmaxf(fmx.x, fmx.y);
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        float s = 0.0f, z = 0.0f;
        if (tv < nv) step_and_zero(mn, mx, qmax, s, z);
        store_meta(blk + o.vm, (jv >> 1) * 32 + tv, c.meta16, s, z, (jv & 1) == 0);
        const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
        // byte tile [c][t] with token t of channel c at t ^ 4 (c / 16): the 8 lanes of a token
        // (channels 16 jv ..) then store into 8 different banks
        const int tsw = tv ^ (jv << 2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 f = PP::f2(w[i]);
            const int ch = 16 * jv + 2 * i;
            uint32_t k0, k1;
            code_pair2(f.x, f.y, s, s, r, r, z, z, (1 << BITS) - 1, k0, k1);
            vc8[ch * kBlockTokens + tsw] = tv < nv ? (uint8_t)k0 : 0;
            vc8[(ch + 1) * kBlockTokens + tsw] = tv < nv ? (uint8_t)k1 : 0;
        }
    }
    __syncthreads();

    // keys: warp w, channel pair cp = 8 w + lane / 4, tokens 8 q .. 8 q + 7 (q = lane & 3)
    {
        const int q = lane & 3, pl = lane >> 2, cp = 8 * warp + pl;
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * q + i;
            w[i] = kt[t * (D / 2) + (cp ^ (q << 3))];
        }
        uint32_t mnp = w[0], mxp = w[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            mnp = PP::mn(mnp, w[i]);
            mxp = PP::mx(mxp, w[i]);
        }
        float2 mn = PP::f2(mnp), mx = PP::f2(mxp);
#pragma unroll
        for (int x = 1; x < 4; x <<= 1) {
            mn.x = fminf(mn.x, __shfl_xor_sync(0xffffffffu, mn.x, x));
            mn.y = fminf(mn.y, __shfl_xor_sync(0xffffffffu, mn.y, x));
            mx.x = fmaxf(mx.x, __shfl_xor_sync(0xffffffffu, mx.x, x));
            mx.y = fmaxf(mx.y, __shfl_xor_sync(0xffffffffu, mx.y, x));
        }
        float s0, z0, s1, z1;
        step_and_zero(mn.x, mx.x, qmax, s0, z0);
        step_and_zero(mn.y, mx.y, qmax, s1, z1);
        store_meta(blk + o.km, 2 * cp, c.meta16, s0, z0, q == 0);
        store_meta(blk + o.km, 2 * cp + 1, c.meta16, s1, z1, q == 0);
        const float r0 = s0 > 0.0f ? __frcp_rn(s0) : 0.0f, r1 = s1 > 0.0f ? __frcp_rn(s1) : 0.0f;
        // INT2: a word holds 16 channels = this warp's 8 pairs (shift 4 pl);
        // INT4: 8 channels = 4 pairs, two words per warp (word pl / 4, shift 8 (pl & 3))
        constexpr int KW = D * BITS / 32;   // code words per key row
        const int shift = BITS == 2 ? 4 * pl : 8 * (pl & 3);
        // after the OR-reduction every lane of a word's group holds the word of token 8 q + i;
        // INT2: lane (pl, q) keeps token 8 q + pl's; INT4: lane (pl, q) keeps tokens
        // 8 q + (pl & 3) and 8 q + (pl & 3) + 4 of word 2 w + pl / 4
        uint32_t mine0 = 0u, mine1 = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = 8 * q + i;
            const float2 f = PP::f2(w[i]);
            uint32_t k0, k1;
            code_pair2(f.x, f.y, s0, s1, r0, r1, z0, z1, (1 << BITS) - 1, k0, k1);
            const uint32_t part0 = t < nv ? (k0 | (k1 << BITS)) << shift : 0u;
            uint32_t part = part0;
            part |= __shfl_xor_sync(0xffffffffu, part, 4);
            part |= __shfl_xor_sync(0xffffffffu, part, 8);
            if (BITS == 2) part |= __shfl_xor_sync(0xffffffffu, part, 16);
            if (BITS == 2) {
                if (pl == i) mine0 = part;
            } else {
                if ((pl & 3) == i) mine0 = part;
                if ((pl & 3) + 4 == i) mine1 = part;
            }
        }
        uint32_t* kc = reinterpret_cast<uint32_t*>(blk + o.kc);
        if (BITS == 2) {
            kc[(8 * q + pl) * KW + warp] = mine0;
        } else {
            kc[(8 * q + (pl & 3)) * KW + 2 * warp + (pl >> 2)] = mine0;
            kc[(8 * q + (pl & 3) + 4) * KW + 2 * warp + (pl >> 2)] = mine1;
        }
    }

    // value code words: channel-major, (32 / BITS) tokens per word
    {
        uint32_t* vw = reinterpret_cast<uint32_t*>(blk + o.vc);
        constexpr int per = 32 / BITS, nw = D * BITS;   // words per block
        for (int e = tid; e < nw; e += kAppendThreads) {
            const int ch = e / BITS, part = e % BITS;
            const uint32_t* row = reinterpret_cast<const uint32_t*>(vc8 + ch * kBlockTokens);
            uint32_t word = 0u;
#pragma unroll
            for (int k = 0; k < per / 4; ++k) {
                // tokens 4 k' .. 4 k' + 3 (k' = part per / 4 + k): one byte each, in word k' ^ (c / 16)
                uint32_t x = row[((part * per / 4) + k) ^ (ch >> 4)];
                if (BITS == 2) {
                    x = (x | (x >> 6)) & 0x000F000Fu;   // b0 | b1 << 2 in byte 0, b2 | b3 << 2 in byte 2
                    x = (x | (x >> 12)) & 0xFFu;        // b0 | b1 << 2 | b2 << 4 | b3 << 6
                    word |= x << (8 * k);
                } else {
                    x = (x | (x >> 4)) & 0x00FF00FFu;   // b0 | b1 << 4 in byte 0, b2 | b3 << 4 in byte 2
                    x = (x | (x >> 8)) & 0xFFFFu;
                    word |= x << (16 * k);
                }
            }
            vw[e] = word;
        }
    }
    if (h == 0 && tid == 0) {
        const long long gi = (long long)b * c.cap_total + c.seg_base[seg] + idx;
        c.blk_len[gi] = nv;
        c.blk_pos[gi] = tok0 + t0;
    }
}

__global__ void dequant_kernel(DevCache c, int n_tok, float* __restrict__ Kout, float* __restrict__ Vout) {
    int flat = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    int seg = 0;
    while (seg < KV_NUM_SEG && flat >= c.n_blocks[seg]) {
        flat -= c.n_blocks[seg];
        ++seg;
    }
    if (seg >= KV_NUM_SEG) return;
    const long long gi = (long long)b * c.cap_total + c.seg_base[seg] + flat;
    const int len = c.blk_len[gi], pos = c.blk_pos[gi];
    const unsigned char* blk = block_ptr(c, b, h, seg, flat);
    const int cls = seg_class(c.kind, seg);
    const int d = c.d;
    const float* cent = c.centroids ? c.centroids + ((long long)b * c.Hkv + h) * d * 4 : nullptr;
    for (int e = threadIdx.x; e < len * d; e += blockDim.x) {
        const int t = e / d, ch = e % d;
        const float2 kv = block_entry(cls, blk, d, c.raw_dtype, c.meta16, cent, t, ch);
        const long long o = (((long long)b * c.Hkv + h) * n_tok + pos + t) * d + ch;
        Kout[o] = kv.x;
        Vout[o] = kv.y;
    }
}

}  // namespace

// K and V rows (fp32, padded), key and value code bytes, and for codebook blocks the
// PSAC basis [d][rp] (fp32)
size_t append_smem_bytes(int d, int rp) {
    return 2 * kBlockTokens * (d + 1) * sizeof(float) + 2 * kBlockTokens * d + (size_t)d * rp * sizeof(float);
}

template <typename T>
static kv_status launch_append_t(const void* K, const void* V, int n_tokens, const kv_cache* cache, int mode,
                                 int uni_seg, const int8_t* win_bits, int n_win, int grid_x, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    if constexpr (sizeof(T) == 2) {
        if (mode == 0 && c.d == kFastD) {
            dim3 grid(grid_x, c.Hkv, c.B);
            if (uni_seg == KV_SEG_INT4)
                append_int128_kernel<T, 4><<<grid, kAppendThreads, 0, st>>>(
                    static_cast<const T*>(K), static_cast<const T*>(V), n_tokens, c, uni_seg, cache->n_tokens);
            else
                append_int128_kernel<T, 2><<<grid, kAppendThreads, 0, st>>>(
                    static_cast<const T*>(K), static_cast<const T*>(V), n_tokens, c, uni_seg, cache->n_tokens);
            return check_launch("append_int128_kernel");
        }
    }
    const size_t sm = append_smem_bytes(c.d, c.kind == KV_CODEBOOK2 ? c.rp : 0);
    const kv_status sa = set_smem_limit(reinterpret_cast<const void*>(append_kernel<T>), 120 * 1024, "append_kernel");
    if (sa != KV_OK) return sa;
    dim3 grid(grid_x, c.Hkv, c.B);
    append_kernel<T><<<grid, kAppendThreads, sm, st>>>(static_cast<const T*>(K), static_cast<const T*>(V), n_tokens,
                                                       c, mode, uni_seg, win_bits, n_win, cache->n_tokens);
    return check_launch("append_kernel");
}

kv_status launch_append(const void* K, const void* V, kv_dtype dt, int n_tokens, const kv_cache* cache, int mode,
                        int uni_seg, const int8_t* win_bits, int n_win, int grid_x, cudaStream_t st) {
    switch (dt) {
        case KV_F32: return launch_append_t<float>(K, V, n_tokens, cache, mode, uni_seg, win_bits, n_win, grid_x, st);
        case KV_F16: return launch_append_t<__half>(K, V, n_tokens, cache, mode, uni_seg, win_bits, n_win, grid_x, st);
        case KV_BF16:
            return launch_append_t<__nv_bfloat16>(K, V, n_tokens, cache, mode, uni_seg, win_bits, n_win, grid_x, st);
    }
    return set_error(KV_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
}

kv_status launch_dequant(const kv_cache* cache, float* Kout, float* Vout, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    const int nb = c.n_blocks[0] + c.n_blocks[1] + c.n_blocks[2];
    if (nb == 0) return KV_OK;
    dim3 grid(nb, c.Hkv, c.B);
    dequant_kernel<<<grid, 256, 0, st>>>(c, cache->n_tokens, Kout, Vout);
    return check_launch("dequant_kernel");
}

}  // namespace bitkv
