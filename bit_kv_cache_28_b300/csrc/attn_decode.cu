// Split-K streaming decode attention: one query token per sequence (n_q == 1)
// over a packed UNIFORM2 / UNIFORM4 / MIXED cache plus the current token(s).
//
// WindowQuant note (何が新しいのか, 技術的に面白い点): during decode the whole
// cache is read once per generated token, so the step is memory-bound; the
// mixed FP16 / INT4 / INT2 cache is stored grouped by bit-width so that each
// class streams contiguously.  This kernel reads every cache byte exactly once.
//
// Work split.  Grid (splits, Hkv, B).  A CTA takes a contiguous, byte-balanced
// range of one (batch, kv head) stream; its 4 warps take blocks w, w+4, ... of
// the range, each block bulk-copied (TMA engine, cp.async.bulk) into the
// warp's own ring of shared-memory slots, several blocks ahead.
//
// Arithmetic.  One warp serves all G = Hq/Hkv (<= 16) query heads of the kv
// head through warp-level m16n8k16 MMAs whose rows are the heads: S = Q K^T
// (keys as columns) and O += P V.  For a quantised block the per-channel key
// step and zero are folded into the query side, q.k_hat = (q o s).code + q.z,
// and the per-token value step and zero into the probability side,
// sum_t p_t v_hat_t = sum_t (p_t s_t) code_t + sum_t p_t z_t, so the B operands
// are the raw codes, turned into exact fp16 integers three instructions per
// pair (byte permute, mask-or of the fp16 exponent, fp16x2 FMA).  RAW16 blocks
// are read with ldmatrix (their chunk-permuted rows are bank-conflict free).
// Products accumulate in fp32.  The Jensen term of "Quantized Keys Steal
// Attention" (abstract) is a per-(block, head) scalar, sum_c q_c^2 s_c^2.
// Current-chunk tokens run on CUDA cores.
//
// Merge.  Warps merge (m, l, o) through shared memory, CTAs write partials,
// and the last CTA of a stream (atomic ticket) merges them:
// m = max m_p, l = sum l_p 2^(m_p - m), o = sum o_p 2^(m_p - m) / l.
#include <cstdio>
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bitkv {

namespace {

using namespace tc;

constexpr int kDW = 4;                    // warps per CTA
constexpr int kDThreads = 32 * kDW;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- warp-level MMA and shared-memory matrix loads ---------------------------
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <typename T>
__device__ __forceinline__ void mma_raw(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) mma_f16(c, a, b0, b1);
    else mma_bf16(c, a, b0, b1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T> __device__ __forceinline__ uint32_t pack_raw(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack_raw<__half>(float lo, float hi) { return pack_f16(lo, hi); }
template <> __device__ __forceinline__ uint32_t pack_raw<__nv_bfloat16>(float lo, float hi) { return pack_bf16(lo, hi); }

template <typename T> __device__ __forceinline__ float2 pair_to_f32(uint32_t w);
template <> __device__ __forceinline__ float2 pair_to_f32<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <> __device__ __forceinline__ float2 pair_to_f32<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Two codes of a packed word as an exact fp16 pair (lower element in the low
// half): select the byte that holds them into both halves, keep each code's
// bits under an fp16 exponent of 2^10 (value 1024 + code * 2^p), then one fp16x2
// FMA removes the 1024 and the 2^p.  Every intermediate is exact.
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t sel, uint32_t mask, uint32_t scale,
                                              uint32_t bias) {
    uint32_t x = __byte_perm(w, 0u, sel);
    x = (x & mask) | 0x64006400u;
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(scale), "r"(bias));
    return r;
}

// Per-lane constants of the code extraction.  MMA fragments pair elements
// (2 tig, 2 tig + 1) and (8 + 2 tig, 8 + 2 tig + 1) of a 16-element k-step;
// in an INT2 word element i sits at bits 2i, in an INT4 word at bits 4i.
struct LaneConst {
    int g, tig;
    uint32_t sel2a, sel2b, mask2, scale2, bias2;
    uint32_t sel4, scale4, bias4;
};

__device__ __forceinline__ LaneConst lane_const(int lane) {
    LaneConst c;
    c.g = lane >> 2;
    c.tig = lane & 3;
    const uint32_t nib = c.tig & 1, b0 = c.tig >> 1, b1 = 2 + (c.tig >> 1);
    c.sel2a = b0 | 0x40u | (b0 << 8) | 0x4000u;
    c.sel2b = b1 | 0x40u | (b1 << 8) | 0x4000u;
    // low half: code at byte bits 4 nib (x 2^(4 nib)); high half: byte bits 2 + 4 nib
    c.mask2 = nib ? 0x00C00030u : 0x000C0003u;
    c.scale2 = nib ? ((0x2400u << 16) | 0x2C00u) : ((0x3400u << 16) | 0x3C00u);   // (2^-4, 2^-6) : (1, 2^-2)
    c.bias2 = nib ? ((0xCC00u << 16) | 0xD400u) : ((0xDC00u << 16) | 0xE400u);    // (-64, -16) : (-1024, -256)
    const uint32_t bt = (uint32_t)c.tig;
    c.sel4 = bt | 0x40u | (bt << 8) | 0x4000u;
    c.scale4 = (0x2C00u << 16) | 0x3C00u;   // (1, 2^-4)
    c.bias4 = (0xD400u << 16) | 0xE400u;    // (-1024, -64)
    return c;
}

// Running softmax state of one warp: rows r = 0 (head g) and r = 1 (head g + 8).
// m in the log2 domain; l and pz are this lane's partial sums (reduced over the
// lane quad at the end); o is the P V accumulator fragment (c0, c1 row g;
// c2, c3 row g + 8) over n-tiles of 8 channels.
template <int D>
struct DecState {
    float m[2], l[2];
    float o[D / 8][4];
    float pz[2][D / 32];
};

template <int D, bool TWO>
__device__ __forceinline__ void online_softmax(DecState<D>& st, float (&x)[2][8], float (&p)[2][8]) {
#pragma unroll
    for (int r = 0; r < (TWO ? 2 : 1); ++r) {
        float mx = x[r][0];
#pragma unroll
        for (int k = 1; k < 8; ++k) mx = fmaxf(mx, x[r][k]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (mx > st.m[r]) {
            const float alpha = ex2(st.m[r] - mx);   // 0 when the old max is -inf
            st.l[r] *= alpha;
#pragma unroll
            for (int jj = 0; jj < D / 8; ++jj) {
                st.o[jj][2 * r] *= alpha;
                st.o[jj][2 * r + 1] *= alpha;
            }
#pragma unroll
            for (int vg = 0; vg < D / 32; ++vg) st.pz[r][vg] *= alpha;
            st.m[r] = mx;
        }
        const float mu = st.m[r] == -INFINITY ? 0.0f : st.m[r];
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            p[r][k] = ex2(x[r][k] - mu);
            s += p[r][k];
        }
        st.l[r] += s;
    }
    if (!TWO) {
#pragma unroll
        for (int k = 0; k < 8; ++k) p[1][k] = 0.0f;
    }
}

__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// ---- one quantised block ------------------------------------------------------
// q[r][4 kk + e]: query of row r at channels 16 kk + 2 tig + {0, 1, 8, 9}.
template <int D, int BITS, bool TWO, int JENSEN>
__device__ __forceinline__ void int_block(const unsigned char* blk, int len, const LaneConst& lc,
                                          const float (&q)[2][D / 4], float c1, float tau, DecState<D>& st) {
    const IntBlockOffsets o = int_offsets(D, BITS);
    // A = q o s as an fp16 pair hi + lo (hi = fp16(q s), lo = fp16(q s - hi): the
    // product keeps ~22 bits, enough for outlier channels with large steps), the
    // zero-point term q.z and the Jensen sum per row
    const float4* km4 = reinterpret_cast<const float4*>(blk + o.km);
    uint32_t aqk[D / 16][4], aql[D / 16][4];
    float qz[2] = {0.0f, 0.0f}, jd[2] = {0.0f, 0.0f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const float4 A = km4[(16 * kk + 2 * lc.tig) >> 1];
        const float4 Bq = km4[(16 * kk + 8 + 2 * lc.tig) >> 1];
        const float s[4] = {A.x, A.z, Bq.x, Bq.z}, z[4] = {A.y, A.w, Bq.y, Bq.w};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (r == 1 && !TWO) {
                aqk[kk][1] = aqk[kk][3] = aql[kk][1] = aql[kk][3] = 0u;
                continue;
            }
            float qs[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qs[e] = q[r][4 * kk + e] * s[e];
                qz[r] = fmaf(q[r][4 * kk + e], z[e], qz[r]);
                if (JENSEN == KV_JENSEN_TAYLOR2) jd[r] = fmaf(qs[e], qs[e], jd[r]);
                else if (JENSEN == KV_JENSEN_EXACT) jd[r] += log_sinhc(0.5f * tau * qs[e]);
            }
            aqk[kk][r] = pack_f16(qs[0], qs[1]);
            aqk[kk][2 + r] = pack_f16(qs[2], qs[3]);
            const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&aqk[kk][r]));
            const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&aqk[kk][2 + r]));
            aql[kk][r] = pack_f16(qs[0] - h01.x, qs[1] - h01.y);
            aql[kk][2 + r] = pack_f16(qs[2] - h23.x, qs[3] - h23.y);
        }
    }
    float bias[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float z = quad_sum(qz[r]);
        float dl = 0.0f;
        if (JENSEN != KV_JENSEN_OFF) {
            dl = quad_sum(jd[r]);
            if (JENSEN == KV_JENSEN_TAYLOR2) dl *= tau * tau * (1.0f / 24.0f);
        }
        bias[r] = (tau * z - dl) * kLog2e;
    }

    // S = (q o s) codes^T
    constexpr int KW = D * BITS / 32;   // code words per key row
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk + o.kc);
    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        uint32_t w[KW];
        const uint4* src = reinterpret_cast<const uint4*>(kc + (8 * j + lc.g) * KW);
#pragma unroll
        for (int i = 0; i < KW / 4; ++i) {
            const uint4 v = src[i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b0, b1;
            if (BITS == 2) {
                b0 = code_pair(w[kk], lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                b1 = code_pair(w[kk], lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                b0 = code_pair(w[2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                b1 = code_pair(w[2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
            mma_f16(acc[j], aqk[kk], b0, b1);
            mma_f16(acc[j], aql[kk], b0, b1);
        }
    }
    float x[2][8], p[2][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool valid = 8 * j + 2 * lc.tig + e < len;
            x[0][2 * j + e] = valid ? fmaf(acc[j][e], c1, bias[0]) : -INFINITY;
            x[1][2 * j + e] = valid ? fmaf(acc[j][2 + e], c1, bias[1]) : -INFINITY;
        }
    online_softmax<D, TWO>(st, x, p);

    // A = p o s_v (fp16) per value group, and the zero-point term sum p z_v
    const float4* vm4 = reinterpret_cast<const float4*>(blk + o.vm);
    uint32_t apv[D / 32][2][4];
#pragma unroll
    for (int vg = 0; vg < D / 32; ++vg)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const float4 SA = vm4[vg * 16 + ((16 * kk + 2 * lc.tig) >> 1)];
            const float4 SB = vm4[vg * 16 + ((16 * kk + 8 + 2 * lc.tig) >> 1)];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r == 1 && !TWO) {
                    apv[vg][kk][1] = apv[vg][kk][3] = 0u;
                    continue;
                }
                const float pa0 = p[r][4 * kk], pa1 = p[r][4 * kk + 1], pb0 = p[r][4 * kk + 2],
                            pb1 = p[r][4 * kk + 3];
                apv[vg][kk][r] = pack_f16(pa0 * SA.x, pa1 * SA.z);
                apv[vg][kk][2 + r] = pack_f16(pb0 * SB.x, pb1 * SB.z);
                st.pz[r][vg] = fmaf(pa0, SA.y, fmaf(pa1, SA.w, fmaf(pb0, SB.y, fmaf(pb1, SB.w, st.pz[r][vg]))));
            }
        }
    // O += (p o s_v) codes
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + o.vc);
#pragma unroll
    for (int jj = 0; jj < D / 8; ++jj) {
        const int ch = 8 * jj + lc.g, vg = jj >> 2;
        if (BITS == 2) {
            const uint2 w = *reinterpret_cast<const uint2*>(vc + ch * 2);
            mma_f16(st.o[jj], apv[vg][0], code_pair(w.x, lc.sel2a, lc.mask2, lc.scale2, lc.bias2),
                    code_pair(w.x, lc.sel2b, lc.mask2, lc.scale2, lc.bias2));
            mma_f16(st.o[jj], apv[vg][1], code_pair(w.y, lc.sel2a, lc.mask2, lc.scale2, lc.bias2),
                    code_pair(w.y, lc.sel2b, lc.mask2, lc.scale2, lc.bias2));
        } else {
            const uint4 w = *reinterpret_cast<const uint4*>(vc + ch * 4);
            mma_f16(st.o[jj], apv[vg][0], code_pair(w.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4),
                    code_pair(w.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4));
            mma_f16(st.o[jj], apv[vg][1], code_pair(w.z, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4),
                    code_pair(w.w, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4));
        }
    }
}

// ---- one RAW16 block (16-bit K and V kept as given) ------------------------------
template <typename T, int D, bool TWO>
__device__ __forceinline__ void raw_block(uint32_t sblk, int len, const LaneConst& lc,
                                          const uint32_t (&aq)[D / 16][4], float c1, DecState<D>& st) {
    const int lane = threadIdx.x & 31, mat = lane >> 3, rr = lane & 7;
    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        const int key = 8 * j + rr;
#pragma unroll
        for (int cq = 0; cq < D / 32; ++cq) {
            const int chunk = 4 * cq + mat;
            uint32_t r0, r1, r2, r3;
            ldsm_x4(sblk + key * (2 * D) + ((chunk ^ rr) << 4), r0, r1, r2, r3);
            mma_raw<T>(acc[j], aq[2 * cq], r0, r1);
            mma_raw<T>(acc[j], aq[2 * cq + 1], r2, r3);
        }
    }
    float x[2][8], p[2][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool valid = 8 * j + 2 * lc.tig + e < len;
            x[0][2 * j + e] = valid ? acc[j][e] * c1 : -INFINITY;
            x[1][2 * j + e] = valid ? acc[j][2 + e] * c1 : -INFINITY;
        }
    online_softmax<D, TWO>(st, x, p);
    uint32_t apv[2][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        apv[kk][0] = pack_raw<T>(p[0][4 * kk], p[0][4 * kk + 1]);
        apv[kk][2] = pack_raw<T>(p[0][4 * kk + 2], p[0][4 * kk + 3]);
        apv[kk][1] = TWO ? pack_raw<T>(p[1][4 * kk], p[1][4 * kk + 1]) : 0u;
        apv[kk][3] = TWO ? pack_raw<T>(p[1][4 * kk + 2], p[1][4 * kk + 3]) : 0u;
    }
    const uint32_t vbase = sblk + kBlockTokens * D * 2;
    const int key = 8 * mat + rr;
#pragma unroll
    for (int jj = 0; jj < D / 8; ++jj) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(vbase + key * (2 * D) + ((jj ^ rr) << 4), r0, r1, r2, r3);
        mma_raw<T>(st.o[jj], apv[0], r0, r1);
        mma_raw<T>(st.o[jj], apv[1], r2, r3);
    }
}

// ---- one unquantised current token, on CUDA cores --------------------------------
template <typename T, int D, bool TWO>
__device__ __forceinline__ void current_token(const T* kr, const T* vr, const LaneConst& lc,
                                              const float (&q)[2][D / 4], float c1, DecState<D>& st) {
    float dot[2] = {0.0f, 0.0f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const float2 ka = pair_to_f32<T>(*reinterpret_cast<const uint32_t*>(kr + 16 * kk + 2 * lc.tig));
        const float2 kb = pair_to_f32<T>(*reinterpret_cast<const uint32_t*>(kr + 16 * kk + 8 + 2 * lc.tig));
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            dot[r] = fmaf(q[r][4 * kk], ka.x, dot[r]);
            dot[r] = fmaf(q[r][4 * kk + 1], ka.y, dot[r]);
            dot[r] = fmaf(q[r][4 * kk + 2], kb.x, dot[r]);
            dot[r] = fmaf(q[r][4 * kk + 3], kb.y, dot[r]);
        }
    }
    float x[2][8], p[2][8];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float s = quad_sum(dot[r]) * c1;
#pragma unroll
        for (int k = 0; k < 8; ++k) x[r][k] = (k == 0 && lc.tig == 0) ? s : -INFINITY;
    }
    online_softmax<D, TWO>(st, x, p);
    float pr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) pr[r] = __shfl_sync(0xffffffffu, p[r][0], (threadIdx.x & 31) & ~3);
#pragma unroll
    for (int jj = 0; jj < D / 8; ++jj) {
        const float2 v = pair_to_f32<T>(*reinterpret_cast<const uint32_t*>(vr + 8 * jj + 2 * lc.tig));
        st.o[jj][0] = fmaf(pr[0], v.x, st.o[jj][0]);
        st.o[jj][1] = fmaf(pr[0], v.y, st.o[jj][1]);
        if (TWO) {
            st.o[jj][2] = fmaf(pr[1], v.x, st.o[jj][2]);
            st.o[jj][3] = fmaf(pr[1], v.y, st.o[jj][3]);
        }
    }
}

// First block of split s of a stream whose blocks (segment-major, RAW16, INT4,
// INT2) are cut into `S` ranges of about equal bytes: the smallest block index
// i with S * (bytes before i) >= s * (total bytes).
__device__ int split_begin(const DevCache& c, int s, int S) {
    long long total = 0;
#pragma unroll
    for (int k = 0; k < KV_NUM_SEG; ++k) total += (long long)c.n_blocks[k] * c.block_bytes[k];
    const long long target = (long long)s * total;
    long long before = 0;
    int base = 0;
#pragma unroll
    for (int k = 0; k < KV_NUM_SEG; ++k) {
        const int n = c.n_blocks[k];
        const long long bb = c.block_bytes[k];
        if (n > 0 && (long long)S * (before + (long long)(n - 1) * bb) >= target) {
            const long long num = target - (long long)S * before;
            const long long j = num <= 0 ? 0 : (num + (long long)S * bb - 1) / ((long long)S * bb);
            return base + (int)j;
        }
        before += (long long)n * bb;
        base += n;
    }
    return base;
}

struct DecShape {
    int nsw;          // ring slots per warp
    int slot_bytes;   // bytes per slot (largest block class of the cache)
    int rows;         // merge rows per warp (8 or 16)
};

template <typename T, int D, bool TWO, int JENSEN>
__global__ void __launch_bounds__(kDThreads, D == 64 ? 3 : 1)
attn_decode_kernel(const T* __restrict__ Q, const T* __restrict__ Kcur, const T* __restrict__ Vcur, int n_cur, int Hq,
                   DevCache c, float tau, int n_splits, DecShape sh, void* __restrict__ out, int out_f32,
                   float* __restrict__ lse, float* __restrict__ part, int* __restrict__ tickets, int* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ volatile int abort_flag;
    __shared__ int s_last;
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = Hq / c.Hkv;
    const int stream = b * c.Hkv + h;
    const LaneConst lc = lane_const(lane);
    const int nsw = sh.nsw, slot_bytes = sh.slot_bytes;
    unsigned char* slots = sm;
    float* mrg = reinterpret_cast<float*>(sm + kDW * nsw * slot_bytes);     // [kDW][rows][D + 2]
    const uint32_t bar0 = smem_u32(mrg + kDW * sh.rows * (D + 2));
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)(warp * nsw + i); };

    if (tid == 0) abort_flag = 0;
    if (lane == 0)
        for (int i = 0; i < nsw; ++i) mbar_init(bar(i), 1);
    mbar_fence_init();
    __syncthreads();

    // queries: fp32 copies for quantised blocks, 16-bit A fragments for RAW16 blocks
    float q[2][D / 4];
    uint32_t aq[D / 16][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int hr = lc.g + 8 * r;
        const bool ok = hr < G && (r == 0 || TWO);
        const T* qrow = Q + ((long long)b * Hq + (long long)h * G + (ok ? hr : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t wa = ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lc.tig) : 0u;
            const uint32_t wb = ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * lc.tig) : 0u;
            const float2 fa = pair_to_f32<T>(wa), fb = pair_to_f32<T>(wb);
            q[r][4 * kk] = fa.x;
            q[r][4 * kk + 1] = fa.y;
            q[r][4 * kk + 2] = fb.x;
            q[r][4 * kk + 3] = fb.y;
            aq[kk][r] = wa;
            aq[kk][2 + r] = wb;
        }
    }
    const float c1 = tau * kLog2e;

    DecState<D> st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.0f;
#pragma unroll
    for (int jj = 0; jj < D / 8; ++jj) st.o[jj][0] = st.o[jj][1] = st.o[jj][2] = st.o[jj][3] = 0.0f;
#pragma unroll
    for (int vg = 0; vg < D / 32; ++vg) st.pz[0][vg] = st.pz[1][vg] = 0.0f;

    // this warp's blocks: lo + warp, lo + warp + kDW, ... below hi
    const int lo = split_begin(c, split, n_splits), hi = split_begin(c, split + 1, n_splits);
    const int nw = lo + warp < hi ? (hi - lo - warp + kDW - 1) / kDW : 0;
    const int n0 = c.n_blocks[0], n01 = c.n_blocks[0] + c.n_blocks[1];
    auto locate = [&](int i, int& seg, int& idx) {
        seg = i < n0 ? 0 : (i < n01 ? 1 : 2);
        idx = i - (seg == 0 ? 0 : (seg == 1 ? n0 : n01));
    };
    auto issue = [&](int k) {
        int seg, idx;
        locate(lo + warp + kDW * k, seg, idx);
        const uint32_t bytes = (uint32_t)c.block_bytes[seg];
        const uint32_t sb = bar(k % nsw);
        mbar_expect_tx(sb, bytes);
        bulk_g2s(smem_u32(slots + (warp * nsw + k % nsw) * slot_bytes), block_ptr(c, b, h, seg, idx), bytes, sb);
    };
    if (lane == 0)
        for (int k = 0; k < nw && k < nsw; ++k) issue(k);
    __syncwarp();
    int k = 0, len_next = 0;
    for (; k < nw; ++k) {
        if ((k & 31) == 0) {
            // valid lengths of the next 32 blocks, one per lane, fetched before the wait
            const int kl = k + lane;
            len_next = 0;
            if (kl < nw) {
                int sg, ix;
                locate(lo + warp + kDW * kl, sg, ix);
                len_next = c.blk_len[(long long)b * c.cap_total + c.seg_base[sg] + ix];
            }
        }
        const bool ok = mbar_wait(bar(k % nsw), (k / nsw) & 1, &abort_flag, err, 1);
        if (!__all_sync(0xffffffffu, ok)) break;
        int seg, idx;
        locate(lo + warp + kDW * k, seg, idx);
        const int len = __shfl_sync(0xffffffffu, len_next, k & 31);
        const unsigned char* blk = slots + (warp * nsw + k % nsw) * slot_bytes;
        const int cls = seg_class(c.kind, seg);
        if (cls == CLS_INT2) int_block<D, 2, TWO, JENSEN>(blk, len, lc, q, c1, tau, st);
        else if (cls == CLS_INT4) int_block<D, 4, TWO, JENSEN>(blk, len, lc, q, c1, tau, st);
        else raw_block<T, D, TWO>(smem_u32(blk), len, lc, aq, c1, st);
        __syncwarp();
        if (lane == 0 && k + nsw < nw) issue(k + nsw);
    }
    if (k < nw && lane == 0) {
        // gave up: let this warp's copies still in flight land (bounded) before the CTA exits
        for (int kk = k; kk < nw && kk < k + nsw; ++kk) {
            const long long t0 = clock64();
            while (!mbar_try_wait(bar(kk % nsw), (kk / nsw) & 1) && clock64() - t0 < 100000000LL) {
            }
        }
    }
    __syncwarp();

    // the current chunk's tokens go to the last split
    if (split == n_splits - 1 && !abort_flag) {
        const long long rbase = (long long)stream * n_cur;
        for (int t = warp; t < n_cur; t += kDW)
            current_token<T, D, TWO>(Kcur + (rbase + t) * D, Vcur + (rbase + t) * D, lc, q, c1, st);
    }

    // finish the lane partial sums and fold the value zero-point term into o
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        st.l[r] = quad_sum(st.l[r]);
#pragma unroll
        for (int vg = 0; vg < D / 32; ++vg) st.pz[r][vg] = quad_sum(st.pz[r][vg]);
    }
#pragma unroll
    for (int jj = 0; jj < D / 8; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[jj][e] += st.pz[e >> 1][jj >> 2];

    // warps -> CTA through shared memory: row layout [m, l, o[0..D)]
    const int rows = sh.rows;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (r == 1 && !TWO) break;
        float* row = mrg + ((warp * rows) + lc.g + 8 * r) * (D + 2);
        if (lc.tig == 0) {
            row[0] = st.m[r];
            row[1] = st.l[r];
        }
#pragma unroll
        for (int jj = 0; jj < D / 8; ++jj) {
            row[2 + 8 * jj + 2 * lc.tig] = st.o[jj][2 * r];
            row[2 + 8 * jj + 2 * lc.tig + 1] = st.o[jj][2 * r + 1];
        }
    }
    __syncthreads();
    const long long rows_out = (long long)c.B * Hq;
    for (int e = tid; e < G * D; e += kDThreads) {
        const int gi = e / D, ch = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDW; ++w) M = fmaxf(M, mrg[(w * rows + gi) * (D + 2)]);
        const float Mu = M == -INFINITY ? 0.0f : M;
        float L = 0.0f, O = 0.0f;
#pragma unroll
        for (int w = 0; w < kDW; ++w) {
            const float* row = mrg + (w * rows + gi) * (D + 2);
            const float f = ex2(row[0] - Mu);
            L = fmaf(row[1], f, L);
            O = fmaf(row[2 + ch], f, O);
        }
        const long long orow = (long long)b * Hq + (long long)h * G + gi;
        if (n_splits == 1) {
            const float v = L > 0.0f ? O / L : 0.0f;
            if (out_f32) static_cast<float*>(out)[orow * D + ch] = v;
            else static_cast<T*>(out)[orow * D + ch] = from_f32<T>(v);
            if (lse && ch == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        } else {
            float* pr = part + (((long long)stream * n_splits + split) * G + gi) * (D + 2);
            if (ch == 0) {
                pr[0] = M;
                pr[1] = L;
            }
            pr[2 + ch] = O;
        }
    }
    (void)rows_out;
    if (n_splits == 1) return;

    // the last CTA of this stream merges every split's partial
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&tickets[stream], 1) == n_splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int e = tid; e < G * D; e += kDThreads) {
        const int gi = e / D, ch = e % D;
        const float* base = part + ((long long)stream * n_splits * G + gi) * (D + 2);
        const long long sstride = (long long)G * (D + 2);
        float M = -INFINITY;
        for (int s = 0; s < n_splits; ++s) {
            const float ls = __ldcg(base + s * sstride + 1);
            if (ls > 0.0f) M = fmaxf(M, __ldcg(base + s * sstride));
        }
        float L = 0.0f, O = 0.0f;
        for (int s = 0; s < n_splits; ++s) {
            const float ls = __ldcg(base + s * sstride + 1);
            if (ls > 0.0f) {
                const float f = ex2(__ldcg(base + s * sstride) - M);
                L = fmaf(ls, f, L);
                O = fmaf(__ldcg(base + s * sstride + 2 + ch), f, O);
            }
        }
        const long long orow = (long long)b * Hq + (long long)h * G + gi;
        const float v = L > 0.0f ? O / L : 0.0f;
        if (out_f32) static_cast<float*>(out)[orow * D + ch] = v;
        else static_cast<T*>(out)[orow * D + ch] = from_f32<T>(v);
        if (lse && ch == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    if (tid == 0) tickets[stream] = 0;
}

int g_dec_sms = 0;
int dec_num_sms() {
    if (g_dec_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_dec_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_dec_sms <= 0) g_dec_sms = 148;
    }
    return g_dec_sms;
}

DecShape dec_shape(const kv_cache* cache, int Hq) {
    const kv_layout& L = cache->layout;
    long long slot = 0;
    for (int s = 0; s < KV_NUM_SEG; ++s)
        if (L.cap_blocks[s] > 0) slot = slot > L.block_bytes[s] ? slot : L.block_bytes[s];
    if (slot == 0) slot = 16;
    DecShape sh;
    sh.slot_bytes = (int)((slot + 127) / 128 * 128);
    int nsw = (int)(64 * 1024 / (kDW * (long long)sh.slot_bytes));
    sh.nsw = nsw < 2 ? 2 : (nsw > 8 ? 8 : nsw);
    sh.rows = Hq / L.Hkv > 8 ? 16 : 8;
    return sh;
}

size_t dec_smem_bytes(const DecShape& sh, int d) {
    return 1024 + (size_t)kDW * sh.nsw * sh.slot_bytes + (size_t)kDW * sh.rows * (d + 2) * sizeof(float) +
           (size_t)kDW * sh.nsw * 8;
}

size_t dec_ticket_bytes(const kv_cache* cache) {
    return ((size_t)cache->layout.B * cache->layout.Hkv * sizeof(int) + 255) / 256 * 256;
}

template <typename T, int D, bool TWO, int JENSEN>
kv_status launch_dec_t(const void* Q, const void* Kc, const void* Vc, int n_cur, int Hq, const kv_cache* cache,
                       float tau, int n_splits, void* out, int out_f32, float* lse, void* ws, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    const DecShape sh = dec_shape(cache, Hq);
    const size_t smem = dec_smem_bytes(sh, D);
    static size_t attr_bytes = 0;
    if (smem > attr_bytes) {
        const cudaError_t e =
            cudaFuncSetAttribute(attn_decode_kernel<T, D, TWO, JENSEN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return set_error(KV_ERR_CUDA, "attn_decode_kernel: %zu bytes of shared memory: %s", smem,
                             cudaGetErrorString(e));
        attr_bytes = smem;
    }
    unsigned char* w = static_cast<unsigned char*>(ws);
    int* err = reinterpret_cast<int*>(w);
    int* tickets = reinterpret_cast<int*>(w + 256);
    float* part = reinterpret_cast<float*>(w + 256 + dec_ticket_bytes(cache));
    cudaMemsetAsync(w, 0, 256 + dec_ticket_bytes(cache), st);
    dim3 grid(n_splits, c.Hkv, c.B);
    attn_decode_kernel<T, D, TWO, JENSEN><<<grid, kDThreads, smem, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(Kc), static_cast<const T*>(Vc), n_cur, Hq, c, tau, n_splits,
        sh, out, out_f32, lse, part, tickets, err);
    kv_status s = check_launch("attn_decode_kernel");
    if (s != KV_OK) return s;
    if (getenv("BITKV_DEBUG_SYNC")) {
        int h_err = 0;
        cudaMemcpyAsync(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost, st);
        cudaStreamSynchronize(st);
        if (h_err) return set_error(KV_ERR_TIMEOUT, "attn_decode_kernel: bounded wait %d gave up", h_err);
    }
    return KV_OK;
}

}  // namespace

bool decode_supported(const kv_cache* cache, kv_dtype dt, int n_q, int Hq) {
    const kv_layout& L = cache->layout;
    if (n_q != 1 || (dt != KV_F16 && dt != KV_BF16)) return false;
    if (L.d != 64 && L.d != 128) return false;
    if (L.kind != KV_UNIFORM2 && L.kind != KV_UNIFORM4 && L.kind != KV_MIXED) return false;
    if (L.kind == KV_MIXED && L.raw_dtype != (int)dt) return false;
    return Hq % L.Hkv == 0 && Hq / L.Hkv <= 16;
}

int decode_auto_splits(const kv_cache* cache, int Hq) {
    const kv_layout& L = cache->layout;
    const DecShape sh = dec_shape(cache, Hq);
    const size_t smem = dec_smem_bytes(sh, L.d);
    int per_sm = (int)((228 * 1024) / (smem + 1024));
    if (per_sm > 16) per_sm = 16;
    if (per_sm < 1) per_sm = 1;
    const int streams = L.B * L.Hkv;
    const int nb = cache->n_blocks[0] + cache->n_blocks[1] + cache->n_blocks[2];
    int s = (per_sm * dec_num_sms()) / (streams > 0 ? streams : 1);
    const int cap = nb / (2 * kDW) > 1 ? nb / (2 * kDW) : 1;   // at least two blocks per warp
    if (s > cap) s = cap;
    return s < 1 ? 1 : s;
}

size_t decode_workspace(const kv_cache* cache, int Hq, int n_splits) {
    const kv_layout& L = cache->layout;
    const int G = Hq / L.Hkv;
    size_t ws = 256 + dec_ticket_bytes(cache);
    if (n_splits > 1) ws += (size_t)L.B * L.Hkv * n_splits * G * (L.d + 2) * sizeof(float);
    return ws;
}

kv_status launch_attn_decode(const void* Q, const void* Kc, const void* Vc, kv_dtype dt, int n_cur, int Hq,
                             const kv_cache* cache, float tau, int jensen, int n_splits, void* out, int out_f32,
                             float* lse, void* ws, cudaStream_t st) {
    const int d = cache->layout.d;
    const bool two = Hq / cache->layout.Hkv > 8;
    using F16 = __half;
    using BF16 = __nv_bfloat16;
#define BITKV_DEC(T, D, TWO)                                                                                    \
    do {                                                                                                        \
        if (jensen == KV_JENSEN_TAYLOR2)                                                                        \
            return launch_dec_t<T, D, TWO, KV_JENSEN_TAYLOR2>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits, out,  \
                                                              out_f32, lse, ws, st);                            \
        if (jensen == KV_JENSEN_EXACT)                                                                          \
            return launch_dec_t<T, D, TWO, KV_JENSEN_EXACT>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits, out,    \
                                                            out_f32, lse, ws, st);                              \
        return launch_dec_t<T, D, TWO, KV_JENSEN_OFF>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits, out, out_f32, \
                                                      lse, ws, st);                                             \
    } while (0)
    if (dt == KV_F16) {
        if (d == 64) { if (two) BITKV_DEC(F16, 64, true); else BITKV_DEC(F16, 64, false); }
        else { if (two) BITKV_DEC(F16, 128, true); else BITKV_DEC(F16, 128, false); }
    } else {
        if (d == 64) { if (two) BITKV_DEC(BF16, 64, true); else BITKV_DEC(BF16, 64, false); }
        else { if (two) BITKV_DEC(BF16, 128, true); else BITKV_DEC(BF16, 128, false); }
    }
#undef BITKV_DEC
}

}  // namespace bitkv
