// Split-K streaming decode attention: one query token per sequence (n_q == 1)
// over a packed UNIFORM2 / UNIFORM4 / MIXED cache plus the current token(s).
//
// WindowQuant note (何が新しいのか, 技術的に面白い点): during decode the whole
// cache is read once per generated token, so the step is memory-bound; the
// mixed FP16 / INT4 / INT2 cache is stored grouped by bit-width so that each
// class streams contiguously.  This kernel reads every cache byte exactly once.
//
// Work split.  A 1-D grid of CTAs over the (batch, kv head) streams, by default one
// wave of resident CTAs (streams past the first (CTAs mod streams) take one split
// fewer).  A CTA takes a contiguous, cost-balanced range of its stream's blocks
// (split_begin); its 4 warps take blocks w, w+4, ... of
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
// pair (byte permute, mask-or of the fp16 exponent, fp16x2 FMA).  Blocks with fp16
// metadata hold fp16 entries, fp16(code s + z): one more fp16x2 FMA forms them exactly
// and they enter the MMAs directly (queries as fp16, the probabilities unscaled).
// RAW16 blocks are read with ldmatrix (their chunk-permuted rows are bank-conflict free).
// Products accumulate in fp32.  The Jensen term of "Quantized Keys Steal
// Attention" (abstract) is a per-(block, head) scalar, sum_c q_c^2 s_c^2.
// Current-chunk tokens run on CUDA cores.
//
// Merge.  Warps merge (m, l, o) through shared memory, CTAs write partials and
// a status word each, and a merge kernel (one CTA per stream, launched with
// programmatic stream serialisation so that it is resident when the decode grid
// ends) combines them, m = max m_p, l = sum l_p 2^(m_p - m), o = sum o_p
// 2^(m_p - m) / l, and writes the call's status header.  Nothing in the workspace
// has to be cleared before a call.
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

// EXACT Jensen terms log(sinh x / x), x = c qs[e], added to acc in the order e = 0 .. 3.  One
// warp vote: when no lane's |x| reaches 1/2, the series alone without branches (the value
// log_sinhc gives there); otherwise log_sinhc per term.  Called by the whole warp.
__device__ __forceinline__ void exact_terms4(float& acc, float c, const float (&qs)[4]) {
    float x[4];
    float xm = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[e] = fabsf(c * qs[e]);
        xm = fmaxf(xm, x[e]);
    }
    if (__any_sync(0xffffffffu, !(xm < 0.5f))) {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc += log_sinhc(x[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) acc += log_sinhc_series(x[e]);
    }
}

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

// Running softmax state of one warp in the transposed form: the MMAs compute
// S^T [keys x heads] and O^T [channels x heads], so a lane owns heads
// 2 tig, 2 tig + 1 (+ 8 nt) of every accumulator fragment.  m in the log2
// domain; l and pz are this lane's partial sums (reduced over the 8 lane
// groups at the end); o[cm][nt] is the O^T fragment of channels 16 cm + g,
// 16 cm + 8 + g.
template <int D, int NT>
struct DecState {
    float m[NT][2], l[NT][2];
    float o[D / 16][NT][4];
    float pz[NT][2][D / 32];
};

__device__ __forceinline__ float group_max(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float group_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    return v + __shfl_xor_sync(0xffffffffu, v, 16);
}
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// x[nt][mt][e]: logits (log2 units) of keys 16 mt + g (e = 0, 1) and 16 mt + 8 + g
// (e = 2, 3) for heads 2 tig + (e & 1) (+ 8 nt).  Updates the running max and sum,
// returns p in the same layout.
template <int D, int NT>
__device__ __forceinline__ void online_softmax(DecState<D, NT>& st, float (&x)[NT][2][4], float (&p)[NT][2][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            float mx = fmaxf(fmaxf(x[nt][0][hc], x[nt][0][2 + hc]), fmaxf(x[nt][1][hc], x[nt][1][2 + hc]));
            mx = group_max(mx);
            if (mx > st.m[nt][hc]) {
                const float alpha = ex2(st.m[nt][hc] - mx);   // 0 when the old max is -inf
                st.l[nt][hc] *= alpha;
#pragma unroll
                for (int cm = 0; cm < D / 16; ++cm) {
                    st.o[cm][nt][hc] *= alpha;
                    st.o[cm][nt][2 + hc] *= alpha;
                }
#pragma unroll
                for (int vg = 0; vg < D / 32; ++vg) st.pz[nt][hc][vg] *= alpha;
                st.m[nt][hc] = mx;
            }
            const float mu = st.m[nt][hc] == -INFINITY ? 0.0f : st.m[nt][hc];
            float s = 0.0f;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float v = ex2(x[nt][mt][2 * r + hc] - mu);
                    p[nt][mt][2 * r + hc] = v;
                    s += v;
                }
            st.l[nt][hc] += s;
        }
}

// ---- one quantised block ------------------------------------------------------
// q[nt][4 kk + e]: query of head g + 8 nt at channels 16 kk + 2 tig + {0, 1, 8, 9}.
template <int D, int BITS, int NT, int JENSEN>
__device__ __forceinline__ void int_block(const unsigned char* blk, int len, const LaneConst& lc,
                                          const float (&q)[NT][D / 4], float c1, float tau, DecState<D, NT>& st) {
    const IntBlockOffsets o = int_offsets(D, BITS, 0);
    // B = (q o s)^T as an fp16 pair hi + lo (hi = fp16(q s), lo = fp16(q s - hi):
    // the product keeps ~22 bits, enough for outlier channels with large steps),
    // the zero-point term q.z and the Jensen sum of head g + 8 nt
    uint32_t bh[NT][D / 16][2], bl[NT][D / 16][2];
    float qz[NT], jd[NT];
    float ss2 = 0.0f;   // ISOTROPIC: sum_c s_c^2 (jd then holds |q|^2)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) qz[nt] = jd[nt] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const float4 A = meta2_at<false>(blk + o.km, 16 * kk + 2 * lc.tig);
        const float4 Bq = meta2_at<false>(blk + o.km, 16 * kk + 8 + 2 * lc.tig);
        const float s[4] = {A.x, A.z, Bq.x, Bq.z}, z[4] = {A.y, A.w, Bq.y, Bq.w};
        if (JENSEN == KV_JENSEN_ISOTROPIC) {
#pragma unroll
            for (int e = 0; e < 4; ++e) ss2 = fmaf(s[e], s[e], ss2);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float qs[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qs[e] = q[nt][4 * kk + e] * s[e];
                qz[nt] = fmaf(q[nt][4 * kk + e], z[e], qz[nt]);
                if (JENSEN == KV_JENSEN_TAYLOR2) jd[nt] = fmaf(qs[e], qs[e], jd[nt]);
                else if (JENSEN == KV_JENSEN_ISOTROPIC) jd[nt] = fmaf(q[nt][4 * kk + e], q[nt][4 * kk + e], jd[nt]);
            }
            if (JENSEN == KV_JENSEN_EXACT) exact_terms4(jd[nt], 0.5f * tau, qs);
            bh[nt][kk][0] = pack_f16(qs[0], qs[1]);
            bh[nt][kk][1] = pack_f16(qs[2], qs[3]);
            const float2 h01 = __half22float2(*reinterpret_cast<const __half2*>(&bh[nt][kk][0]));
            const float2 h23 = __half22float2(*reinterpret_cast<const __half2*>(&bh[nt][kk][1]));
            bl[nt][kk][0] = pack_f16(qs[0] - h01.x, qs[1] - h01.y);
            bl[nt][kk][1] = pack_f16(qs[2] - h23.x, qs[3] - h23.y);
        }
    }
    // bias of head g + 8 nt, then gathered for the fragment's heads 2 tig, 2 tig + 1
    float bias[NT][2];
    const float ms2 = JENSEN == KV_JENSEN_ISOTROPIC ? quad_sum(ss2) * (1.0f / D) : 0.0f;   // mean_c s_c^2
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float dl = 0.0f;
        if (JENSEN != KV_JENSEN_OFF) {
            dl = quad_sum(jd[nt]);
            if (JENSEN == KV_JENSEN_TAYLOR2) dl *= tau * tau * (1.0f / 24.0f);
            else if (JENSEN == KV_JENSEN_ISOTROPIC) dl = tau * tau * (1.0f / 24.0f) * dl * ms2;
        }
        const float bq = (tau * quad_sum(qz[nt]) - dl) * kLog2e;
        bias[nt][0] = __shfl_sync(0xffffffffu, bq, (2 * lc.tig) << 2);
        bias[nt][1] = __shfl_sync(0xffffffffu, bq, (2 * lc.tig + 1) << 2);
    }

    // S^T = codes (q o s)^T: A = key codes [16 keys x 16 channels] per (mt, kk)
    constexpr int KW = D * BITS / 32;   // code words per key row
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk + o.kc);
    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        uint32_t wa[KW], wb[KW];
        const uint4* sa = reinterpret_cast<const uint4*>(kc + (16 * mt + lc.g) * KW);
        const uint4* sb = reinterpret_cast<const uint4*>(kc + (16 * mt + 8 + lc.g) * KW);
#pragma unroll
        for (int i = 0; i < KW / 4; ++i) {
            const uint4 va = sa[i], vb = sb[i];
            wa[4 * i] = va.x; wa[4 * i + 1] = va.y; wa[4 * i + 2] = va.z; wa[4 * i + 3] = va.w;
            wb[4 * i] = vb.x; wb[4 * i + 1] = vb.y; wb[4 * i + 2] = vb.z; wb[4 * i + 3] = vb.w;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            if (BITS == 2) {
                a[0] = code_pair(wa[kk], lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[1] = code_pair(wb[kk], lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[2] = code_pair(wa[kk], lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                a[3] = code_pair(wb[kk], lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                a[0] = code_pair(wa[2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[1] = code_pair(wb[2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[2] = code_pair(wa[2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[3] = code_pair(wb[2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma_f16(acc[mt][nt], a, bh[nt][kk][0], bh[nt][kk][1]);
                mma_f16(acc[mt][nt], a, bl[nt][kk][0], bl[nt][kk][1]);
            }
        }
    }
    float x[NT][2][4], p[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = 16 * mt + 8 * (e >> 1) + lc.g < len;
                x[nt][mt][e] = valid ? fmaf(acc[mt][nt][e], c1, bias[nt][e & 1]) : -INFINITY;
            }
    online_softmax<D, NT>(st, x, p);

    // B = (p o s_v) per value group, transposed to [keys x heads] by movmatrix,
    // and the zero-point term sum p z_v
    uint32_t bpv[D / 32][NT][2][2];
#pragma unroll
    for (int vg = 0; vg < D / 32; ++vg)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float2 sz = meta_at<false>(blk + o.vm, vg * 32 + 16 * mt + 8 * r + lc.g);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float p0 = p[nt][mt][2 * r], p1 = p[nt][mt][2 * r + 1];
                    bpv[vg][nt][mt][r] = movmatrix_t(pack_f16(p0 * sz.x, p1 * sz.x));
                    st.pz[nt][0][vg] = fmaf(p0, sz.y, st.pz[nt][0][vg]);
                    st.pz[nt][1][vg] = fmaf(p1, sz.y, st.pz[nt][1][vg]);
                }
            }
    // O^T += value codes [16 channels x 16 keys] (p o s_v)
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + o.vc);
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm) {
        const int ca = 16 * cm + lc.g, cb = ca + 8, vg = cm >> 1;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t a[4];
            if (BITS == 2) {
                const uint32_t wa = vc[ca * 2 + kk], wb = vc[cb * 2 + kk];
                a[0] = code_pair(wa, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[1] = code_pair(wb, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[2] = code_pair(wa, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                a[3] = code_pair(wb, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                const uint2 wa = *reinterpret_cast<const uint2*>(vc + ca * 4 + 2 * kk);
                const uint2 wb = *reinterpret_cast<const uint2*>(vc + cb * 4 + 2 * kk);
                a[0] = code_pair(wa.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[1] = code_pair(wb.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[2] = code_pair(wa.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[3] = code_pair(wb.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(st.o[cm][nt], a, bpv[vg][nt][kk][0], bpv[vg][nt][kk][1]);
        }
    }
}

// ---- one quantised block with fp16 metadata ---------------------------------------
// The cache's entries are fp16 numbers, x_hat = fp16(code s + z) with one rounding, so
// they are formed here exactly (fp16x2 FMA of the exact fp16 codes with the channel or
// token (s, z) pairs) and enter the MMAs as they are: S^T = K_hat q^T with the queries as
// fp16 (exact for fp16 I/O and for bf16 values in the fp16 normal range), and
// O^T += V_hat^T p.  The Jensen sum still reads the key steps.
template <int D, int BITS, int NT, int JENSEN>
__device__ __forceinline__ void int_block_h(const unsigned char* blk, int len, const LaneConst& lc,
                                            const float (&q)[NT][D / 4], float c1, float tau, DecState<D, NT>& st) {
    const IntBlockOffsets o = int_offsets(D, BITS, 1);
    const uint32_t* km = reinterpret_cast<const uint32_t*>(blk + o.km);   // channel c: (s_c, z_c)
    // per k-step: (s, s) and (z, z) of the lane's channel pairs 2 tig and 8 + 2 tig
    uint32_t sp[D / 16][2], zp[D / 16][2];
    uint32_t bq[NT][D / 16][2];
    float jd[NT];
    float ss2 = 0.0f;   // ISOTROPIC: sum_c s_c^2 (jd then holds |q|^2)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) jd[nt] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const uint2 m = *reinterpret_cast<const uint2*>(km + 16 * kk + 8 * hf + 2 * lc.tig);
            sp[kk][hf] = __byte_perm(m.x, m.y, 0x5410);
            zp[kk][hf] = __byte_perm(m.x, m.y, 0x7632);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            bq[nt][kk][0] = pack_f16(q[nt][4 * kk], q[nt][4 * kk + 1]);
            bq[nt][kk][1] = pack_f16(q[nt][4 * kk + 2], q[nt][4 * kk + 3]);
        }
        if (JENSEN != KV_JENSEN_OFF) {
            const float2 s01 = __half22float2(*reinterpret_cast<const __half2*>(&sp[kk][0]));
            const float2 s23 = __half22float2(*reinterpret_cast<const __half2*>(&sp[kk][1]));
            const float s[4] = {s01.x, s01.y, s23.x, s23.y};
            if (JENSEN == KV_JENSEN_ISOTROPIC) {
#pragma unroll
                for (int e = 0; e < 4; ++e) ss2 = fmaf(s[e], s[e], ss2);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float qs[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qs[e] = q[nt][4 * kk + e] * s[e];
                    if (JENSEN == KV_JENSEN_TAYLOR2) jd[nt] = fmaf(qs[e], qs[e], jd[nt]);
                    else if (JENSEN == KV_JENSEN_ISOTROPIC) jd[nt] = fmaf(q[nt][4 * kk + e], q[nt][4 * kk + e], jd[nt]);
                }
                if (JENSEN == KV_JENSEN_EXACT) exact_terms4(jd[nt], 0.5f * tau, qs);
            }
        }
    }
    // the Jensen bias of head g + 8 nt, gathered for the fragment's heads 2 tig, 2 tig + 1
    float bias[NT][2];
    const float ms2 = JENSEN == KV_JENSEN_ISOTROPIC ? quad_sum(ss2) * (1.0f / D) : 0.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float dl = 0.0f;
        if (JENSEN != KV_JENSEN_OFF) {
            dl = quad_sum(jd[nt]);
            if (JENSEN == KV_JENSEN_TAYLOR2) dl *= tau * tau * (1.0f / 24.0f);
            else if (JENSEN == KV_JENSEN_ISOTROPIC) dl = tau * tau * (1.0f / 24.0f) * dl * ms2;
        }
        const float bq0 = -dl * kLog2e;
        bias[nt][0] = __shfl_sync(0xffffffffu, bq0, (2 * lc.tig) << 2);
        bias[nt][1] = __shfl_sync(0xffffffffu, bq0, (2 * lc.tig + 1) << 2);
    }

    constexpr int KW = D * BITS / 32;   // code words per key row
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk + o.kc);
    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        uint32_t wa[KW], wb[KW];
        const uint4* sa = reinterpret_cast<const uint4*>(kc + (16 * mt + lc.g) * KW);
        const uint4* sb = reinterpret_cast<const uint4*>(kc + (16 * mt + 8 + lc.g) * KW);
#pragma unroll
        for (int i = 0; i < KW / 4; ++i) {
            const uint4 va = sa[i], vb = sb[i];
            wa[4 * i] = va.x; wa[4 * i + 1] = va.y; wa[4 * i + 2] = va.z; wa[4 * i + 3] = va.w;
            wb[4 * i] = vb.x; wb[4 * i + 1] = vb.y; wb[4 * i + 2] = vb.z; wb[4 * i + 3] = vb.w;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            if (BITS == 2) {
                a[0] = code_pair(wa[kk], lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[1] = code_pair(wb[kk], lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[2] = code_pair(wa[kk], lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                a[3] = code_pair(wb[kk], lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                a[0] = code_pair(wa[2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[1] = code_pair(wb[2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[2] = code_pair(wa[2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[3] = code_pair(wb[2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
            a[0] = hfma2_u32(a[0], sp[kk][0], zp[kk][0]);
            a[1] = hfma2_u32(a[1], sp[kk][0], zp[kk][0]);
            a[2] = hfma2_u32(a[2], sp[kk][1], zp[kk][1]);
            a[3] = hfma2_u32(a[3], sp[kk][1], zp[kk][1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(acc[mt][nt], a, bq[nt][kk][0], bq[nt][kk][1]);
        }
    }
    float x[NT][2][4], p[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = 16 * mt + 8 * (e >> 1) + lc.g < len;
                x[nt][mt][e] = valid ? fmaf(acc[mt][nt][e], c1, bias[nt][e & 1]) : -INFINITY;
            }
    online_softmax<D, NT>(st, x, p);

    // B = p transposed to [keys x heads] by movmatrix (pad keys: p = 0)
    uint32_t bp[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) bp[nt][mt][r] = movmatrix_t(pack_f16(p[nt][mt][2 * r], p[nt][mt][2 * r + 1]));
    // O^T += V_hat [16 channels x 16 keys] p: tokens 16 kk + 2 tig (+ 8) of value group vg
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + o.vc);
    const uint32_t* vm = reinterpret_cast<const uint32_t*>(blk + o.vm);   // (group, token): (s, z)
#pragma unroll
    for (int vg = 0; vg < D / 32; ++vg)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t vs[2], vz[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint2 m = *reinterpret_cast<const uint2*>(vm + vg * 32 + 16 * kk + 8 * hf + 2 * lc.tig);
                vs[hf] = __byte_perm(m.x, m.y, 0x5410);
                vz[hf] = __byte_perm(m.x, m.y, 0x7632);
            }
#pragma unroll
            for (int cm = 2 * vg; cm < 2 * vg + 2; ++cm) {
                const int ca = 16 * cm + lc.g, cb = ca + 8;
                uint32_t a[4];
                if (BITS == 2) {
                    const uint32_t wa = vc[ca * 2 + kk], wb = vc[cb * 2 + kk];
                    a[0] = code_pair(wa, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                    a[1] = code_pair(wb, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                    a[2] = code_pair(wa, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                    a[3] = code_pair(wb, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                } else {
                    const uint2 wa = *reinterpret_cast<const uint2*>(vc + ca * 4 + 2 * kk);
                    const uint2 wb = *reinterpret_cast<const uint2*>(vc + cb * 4 + 2 * kk);
                    a[0] = code_pair(wa.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                    a[1] = code_pair(wb.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                    a[2] = code_pair(wa.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                    a[3] = code_pair(wb.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                }
                a[0] = hfma2_u32(a[0], vs[0], vz[0]);
                a[1] = hfma2_u32(a[1], vs[0], vz[0]);
                a[2] = hfma2_u32(a[2], vs[1], vz[1]);
                a[3] = hfma2_u32(a[3], vs[1], vz[1]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_f16(st.o[cm][nt], a, bp[nt][kk][0], bp[nt][kk][1]);
            }
        }
}

// ---- one RAW16 block (16-bit K and V kept as given) ------------------------------
template <typename T, int D, int NT>
__device__ __forceinline__ void raw_block(uint32_t sblk, int len, const LaneConst& lc,
                                          const uint32_t (&aq)[NT][D / 16][2], float c1, DecState<D, NT>& st) {
    const int lane = threadIdx.x & 31, mat = lane >> 3, rr = lane & 7;
    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;
        const int key = 16 * mt + 8 * (mat & 1) + rr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int chunk = 2 * kk + (mat >> 1);
            uint32_t a[4];
            ldsm_x4(sblk + key * (2 * D) + ((chunk ^ rr) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_raw<T>(acc[mt][nt], a, aq[nt][kk][0], aq[nt][kk][1]);
        }
    }
    float x[NT][2][4], p[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool valid = 16 * mt + 8 * (e >> 1) + lc.g < len;
                x[nt][mt][e] = valid ? acc[mt][nt][e] * c1 : -INFINITY;
            }
    online_softmax<D, NT>(st, x, p);
    uint32_t bpv[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) bpv[nt][mt][r] = movmatrix_t(pack_raw<T>(p[nt][mt][2 * r], p[nt][mt][2 * r + 1]));
    const uint32_t vbase = sblk + kBlockTokens * D * 2;
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const int key = 16 * kk + 8 * (mat >> 1) + rr, chunk = 2 * cm + (mat & 1);
            uint32_t a[4];
            ldsm_x4_t(vbase + key * (2 * D) + ((chunk ^ rr) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_raw<T>(st.o[cm][nt], a, bpv[nt][kk][0], bpv[nt][kk][1]);
        }
}

// ---- one unquantised current token, on CUDA cores --------------------------------
template <typename T, int D, int NT>
__device__ __forceinline__ void current_token(const T* kr, const T* vr, const LaneConst& lc,
                                              const float (&q)[NT][D / 4], float c1, DecState<D, NT>& st) {
    float x[NT][2][4], p[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float dot = 0.0f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const float2 ka = pair_to_f32<T>(*reinterpret_cast<const uint32_t*>(kr + 16 * kk + 2 * lc.tig));
            const float2 kb = pair_to_f32<T>(*reinterpret_cast<const uint32_t*>(kr + 16 * kk + 8 + 2 * lc.tig));
            dot = fmaf(q[nt][4 * kk], ka.x, dot);
            dot = fmaf(q[nt][4 * kk + 1], ka.y, dot);
            dot = fmaf(q[nt][4 * kk + 2], kb.x, dot);
            dot = fmaf(q[nt][4 * kk + 3], kb.y, dot);
        }
        const float s = quad_sum(dot) * c1;    // head g + 8 nt, in every lane of the quad
        const float s0 = __shfl_sync(0xffffffffu, s, (2 * lc.tig) << 2);
        const float s1 = __shfl_sync(0xffffffffu, s, (2 * lc.tig + 1) << 2);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) x[nt][mt][e] = -INFINITY;
        if (lc.g == 0) {           // the token sits in key slot 0 of the lane group g = 0
            x[nt][0][0] = s0;
            x[nt][0][1] = s1;
        }
    }
    online_softmax<D, NT>(st, x, p);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float p0 = __shfl_sync(0xffffffffu, p[nt][0][0], lc.tig);
        const float p1 = __shfl_sync(0xffffffffu, p[nt][0][1], lc.tig);
#pragma unroll
        for (int cm = 0; cm < D / 16; ++cm) {
            const float va = to_f32<T>(vr[16 * cm + lc.g]), vb = to_f32<T>(vr[16 * cm + 8 + lc.g]);
            st.o[cm][nt][0] = fmaf(p0, va, st.o[cm][nt][0]);
            st.o[cm][nt][1] = fmaf(p1, va, st.o[cm][nt][1]);
            st.o[cm][nt][2] = fmaf(p0, vb, st.o[cm][nt][2]);
            st.o[cm][nt][3] = fmaf(p1, vb, st.o[cm][nt][3]);
        }
    }
}

// First block of split s of a stream (segment-major: RAW16, INT4, INT2 blocks) cut into
// S ranges of equal cost.  A warp's time per block, measured with all three classes
// resident: RAW16 0.7, INT4 1.13 and INT2 1 times that of an INT2 block (an 8 KB RAW16
// block streams 4x the bytes of a 2 KB INT2 block but issues about a third of its
// instructions; an INT4 block has twice the codes of an INT2 block).  Hence the weights
// 7 : 11 : 10 per block; split s starts at the first block where the running cost
// reaches s / S of the stream's total.
__device__ __forceinline__ int split_begin(const DevCache& c, int s, int S) {
    long long w[KV_NUM_SEG], total = 0;
#pragma unroll
    for (int g = 0; g < KV_NUM_SEG; ++g) {
        const int cls = seg_class(c.kind, g);
        w[g] = cls == CLS_INT2 ? 10 : (cls == CLS_INT4 ? 11 : 7);
        total += w[g] * c.n_blocks[g];
    }
    const long long t = (long long)s * total / S;
    long long acc = 0;
    int first = 0;
#pragma unroll
    for (int g = 0; g < KV_NUM_SEG; ++g) {
        const long long span = w[g] * c.n_blocks[g];
        if (t <= acc + span) return first + (int)((t - acc + w[g] - 1) / w[g]);
        acc += span;
        first += c.n_blocks[g];
    }
    return first;
}

// Split of CTA i of a grid of n_ctas CTAs over `streams` (batch, kv head) streams: the
// first n_ctas % streams streams take one split more than the others, so that a grid of
// exactly the resident CTA count keeps every SM at the same number of CTAs.
struct SplitOf {
    int stream, split, n;
};
__device__ __forceinline__ SplitOf split_of(int i, int n_ctas, int streams) {
    const int base = n_ctas / streams, extra = n_ctas % streams;
    SplitOf r;
    if (i < extra * (base + 1)) {
        r.stream = i / (base + 1);
        r.split = i % (base + 1);
        r.n = base + 1;
    } else {
        const int k = i - extra * (base + 1);
        r.stream = extra + k / base;
        r.split = k % base;
        r.n = base;
    }
    return r;
}

// Programmatic dependent launch (sm_90 and later): a grid launched with programmatic
// stream serialisation may start while the previous grid of its stream runs, once every
// CTA of that grid has executed launch_dependents; griddep_wait() returns when the
// previous grid has completed and its memory writes are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr int kMergeSmemFloats = 12288;   // the merge kernel's shared-memory weights (48 KB at most)

struct DecShape {
    int nsw;          // ring slots per warp
    int slot_bytes;   // bytes per slot (largest block class of the cache)
    int rows;         // merge rows per warp (8 or 16)
};

template <typename T, int D, int NT, int JENSEN, bool M16>
__global__ void __launch_bounds__(kDThreads, (D == 64 && NT == 1) ? 4 : ((D == 128 && NT == 2) ? 1 : 2))
attn_decode_kernel(const T* __restrict__ Q, const T* __restrict__ Kcur, const T* __restrict__ Vcur, int n_cur, int Hq,
                   DevCache c, float tau, int max_splits, int n_ctas, DecShape sh, void* __restrict__ out, int out_f32,
                   float* __restrict__ lse, float* __restrict__ part, int* __restrict__ cta_status, int stall) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ volatile int abort_flag;
    __shared__ int s_code, s_range;
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA's stream and split; partial rows are laid out with max_splits per stream
    const SplitOf so = split_of(blockIdx.x, n_ctas, c.B * c.Hkv);
    const int split = so.split, n_splits = so.n, stream = so.stream;
    const int h = stream % c.Hkv, b = stream / c.Hkv;
    const int G = Hq / c.Hkv;
    const LaneConst lc = lane_const(lane);
    const int nsw = sh.nsw, slot_bytes = sh.slot_bytes;
    unsigned char* slots = sm;
    float* mrg = reinterpret_cast<float*>(sm + kDW * nsw * slot_bytes);     // [kDW][rows][D + 2]
    const uint32_t bar0 = smem_u32(mrg + kDW * sh.rows * (D + 2));
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)(warp * nsw + i); };

    // bar0 + 8 kDW nsw: a barrier nothing arrives on, the target of the injected stall
    // (failure tests)
    if (tid == 0) {
        abort_flag = 0;
        s_code = s_range = 0;
        mbar_init(bar0 + 8u * (uint32_t)(kDW * nsw), 1);
    }
    if (lane == 0)
        for (int i = 0; i < nsw; ++i) mbar_init(bar(i), 1);
    mbar_fence_init();
    __syncthreads();
    // the merge grid that follows may be scheduled from now on (it waits for this grid)
    griddep_launch_dependents();

    // queries of head g + 8 nt: fp32 copies for quantised blocks, 16-bit B fragments
    // (channel pairs 2 tig, 8 + 2 tig of each k-step) for RAW16 blocks
    float q[NT][D / 4];
    uint32_t aq[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int hr = lc.g + 8 * nt;
        const bool ok = hr < G;
        const T* qrow = Q + ((long long)b * Hq + (long long)h * G + (ok ? hr : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t wa = ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * lc.tig) : 0u;
            const uint32_t wb = ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * lc.tig) : 0u;
            const float2 fa = pair_to_f32<T>(wa), fb = pair_to_f32<T>(wb);
            q[nt][4 * kk] = fa.x;
            q[nt][4 * kk + 1] = fa.y;
            q[nt][4 * kk + 2] = fb.x;
            q[nt][4 * kk + 3] = fb.y;
            aq[nt][kk][0] = wa;
            aq[nt][kk][1] = wb;
        }
    }
    if constexpr (M16 && !std::is_same<T, __half>::value) {
        // fp16-metadata blocks take the queries as fp16: flag any beyond its range
        bool bad = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < D / 4; ++e) bad |= !(fabsf(q[nt][e]) < 65520.0f);
        if (__any_sync(0xffffffffu, bad) && lane == 0) s_range = 1;
    }
    const float c1 = tau * kLog2e;

    DecState<D, NT> st;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        st.m[nt][0] = st.m[nt][1] = -INFINITY;
        st.l[nt][0] = st.l[nt][1] = 0.0f;
#pragma unroll
        for (int cm = 0; cm < D / 16; ++cm) st.o[cm][nt][0] = st.o[cm][nt][1] = st.o[cm][nt][2] = st.o[cm][nt][3] = 0.0f;
#pragma unroll
        for (int vg = 0; vg < D / 32; ++vg) st.pz[nt][0][vg] = st.pz[nt][1][vg] = 0.0f;
    }

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
        // (failure tests: with `stall` the first wait targets a barrier nothing arrives on,
        // with a short limit, so the bounded-wait abort path runs)
        const bool ok = stall && k == 0
                            ? mbar_wait(bar0 + 8u * (uint32_t)(kDW * nsw), 0, &abort_flag, nullptr, 12, 1LL << 21)
                            : mbar_wait(bar(k % nsw), (k / nsw) & 1, &abort_flag, nullptr, 1);
        if (!__all_sync(0xffffffffu, ok)) {
            // a wait gave up here or in another warp: the status word gets the wait's code
            if (lane == 0) atomicCAS(&s_code, 0, stall && k == 0 ? 12 : 1);
            break;
        }
        int seg, idx;
        locate(lo + warp + kDW * k, seg, idx);
        const int len = __shfl_sync(0xffffffffu, len_next, k & 31);
        const unsigned char* blk = slots + (warp * nsw + k % nsw) * slot_bytes;
        const int cls = seg_class(c.kind, seg);
        if (M16 && cls == CLS_INT2) int_block_h<D, 2, NT, JENSEN>(blk, len, lc, q, c1, tau, st);
        else if (M16 && cls == CLS_INT4) int_block_h<D, 4, NT, JENSEN>(blk, len, lc, q, c1, tau, st);
        else if (cls == CLS_INT2) int_block<D, 2, NT, JENSEN>(blk, len, lc, q, c1, tau, st);
        else if (cls == CLS_INT4) int_block<D, 4, NT, JENSEN>(blk, len, lc, q, c1, tau, st);
        else raw_block<T, D, NT>(smem_u32(blk), len, lc, aq, c1, st);
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
            current_token<T, D, NT>(Kcur + (rbase + t) * D, Vcur + (rbase + t) * D, lc, q, c1, st);
    }

    // finish the lane partial sums (over the 8 lane groups) and fold the value
    // zero-point term into o
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            st.l[nt][hc] = group_sum(st.l[nt][hc]);
#pragma unroll
            for (int vg = 0; vg < D / 32; ++vg) st.pz[nt][hc][vg] = group_sum(st.pz[nt][hc][vg]);
        }
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[cm][nt][e] += st.pz[nt][e & 1][cm >> 1];

    // warps -> CTA through shared memory: row (head) layout [m, l, o[0..D)]
    const int rows = sh.rows;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            float* row = mrg + ((warp * rows) + 2 * lc.tig + hc + 8 * nt) * (D + 2);
            if (lc.g == 0) {
                row[0] = st.m[nt][hc];
                row[1] = st.l[nt][hc];
            }
#pragma unroll
            for (int cm = 0; cm < D / 16; ++cm) {
                row[2 + 16 * cm + lc.g] = st.o[cm][nt][hc];
                row[2 + 16 * cm + 8 + lc.g] = st.o[cm][nt][2 + hc];
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
            float* pr = part + (((long long)stream * max_splits + split) * G + gi) * (D + 4);
            if (ch == 0) {
                pr[0] = M;
                pr[1] = L;
            }
            pr[4 + ch] = O;
        }
    }
    (void)rows_out;
    // this CTA's status word, written on every call (the merge kernel folds the words of all
    // CTAs into the status header): the code of a wait that gave up, bit 16 the range flag
    if (tid == 0) cta_status[blockIdx.x] = s_code | (s_range << 16);
}


// Merge of the split partials of one (batch, kv head) stream into its G output rows:
// m = max m_s, l = sum l_s 2^(m_s - m), o = sum o_s 2^(m_s - m) / l.  Partial rows are
// (m, l, -, -, o[D]) in D + 4 floats (o 16-byte aligned), split-major.  Up to 16 splits
// every thread loads all (m, l) pairs and its 16-byte partials together; more splits go
// through shared-memory weights (when smem_floats holds them) or plain loops.
template <typename T, int D>
__device__ __forceinline__ void merge_splits(const float* __restrict__ pbase, int n_splits, int G, int b, int h,
                                             int Hq, float* smem, int smem_floats, void* __restrict__ out,
                                             int out_f32, float* __restrict__ lse, int tid) {
    // partial rows are (m, l, -, -, o[D]): D + 4 floats, o 16-byte aligned
    float* mls = smem;                         // [n_splits * G] (m, l)
    float* fws = mls + 2 * n_splits * G;       // [n_splits * G] weights 2^(m_s - m)
    float* hml = fws + n_splits * G;           // [G] (m, l) of the merged rows
    constexpr int kC4 = D / 4;
    const long long sstride4 = (long long)G * (D + 4) / 4;
    if (n_splits <= 16) {
        // each thread takes (head, 4-channel group) slots; every split's (m, l) and the
        // first 8 splits' 16-byte partials load together, the other 8 in a second round;
        // the thread forms the weights itself
        for (int e = tid; e < G * kC4; e += kDThreads) {
            const int gi = e / kC4, c4 = e % kC4;
            const float* row0 = pbase + (long long)gi * (D + 4);
            const float4* o0 = reinterpret_cast<const float4*>(row0 + 4) + c4;
            float2 ml[16];
            float4 o[8];
#pragma unroll
            for (int sp = 0; sp < 16; ++sp)
                ml[sp] = sp < n_splits ? __ldcg(reinterpret_cast<const float2*>(row0 + sp * sstride4 * 4))
                                       : make_float2(-INFINITY, 0.0f);
#pragma unroll
            for (int sp = 0; sp < 8; ++sp)
                o[sp] = sp < n_splits ? __ldcg(o0 + sp * sstride4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float M = -INFINITY;
#pragma unroll
            for (int sp = 0; sp < 16; ++sp)
                if (ml[sp].y > 0.0f) M = fmaxf(M, ml[sp].x);
            float L = 0.0f;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                if (half == 1) {
#pragma unroll
                    for (int sp = 0; sp < 8; ++sp)
                        o[sp] = 8 + sp < n_splits ? __ldcg(o0 + (8 + sp) * sstride4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
#pragma unroll
                for (int sp = 0; sp < 8; ++sp) {
                    const float2 w = ml[8 * half + sp];
                    const float f = w.y > 0.0f ? ex2(w.x - M) : 0.0f;
                    L = fmaf(w.y, f, L);
                    acc.x = fmaf(o[sp].x, f, acc.x);
                    acc.y = fmaf(o[sp].y, f, acc.y);
                    acc.z = fmaf(o[sp].z, f, acc.z);
                    acc.w = fmaf(o[sp].w, f, acc.w);
                }
            }
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;
            const long long orow = (long long)b * Hq + (long long)h * G + gi;
            const float v[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
            if (out_f32) {
                reinterpret_cast<float4*>(static_cast<float*>(out) + orow * D)[c4] = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                T* dst = static_cast<T*>(out) + orow * D + 4 * c4;
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = from_f32<T>(v[k]);
            }
            if (lse && c4 == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    } else if (3 * n_splits * G + 2 * G <= smem_floats) {
        for (int e = tid; e < n_splits * G; e += kDThreads) {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(pbase + (long long)e * (D + 4)));
            mls[2 * e] = v.x;
            mls[2 * e + 1] = v.y;
        }
        __syncthreads();
        for (int gi = tid; gi < G; gi += kDThreads) {
            float M = -INFINITY;
            for (int sp = 0; sp < n_splits; ++sp)
                if (mls[2 * (sp * G + gi) + 1] > 0.0f) M = fmaxf(M, mls[2 * (sp * G + gi)]);
            float L = 0.0f;
            for (int sp = 0; sp < n_splits; ++sp) {
                const float ls = mls[2 * (sp * G + gi) + 1];
                const float f = ls > 0.0f ? ex2(mls[2 * (sp * G + gi)] - M) : 0.0f;
                fws[sp * G + gi] = f;
                L = fmaf(ls, f, L);
            }
            hml[2 * gi] = M;
            hml[2 * gi + 1] = L;
        }
        __syncthreads();
        // thread -> (head, 4-channel group), weights from shared memory; empty splits
        // carry f = 0 and o = 0
        for (int e = tid; e < G * kC4; e += kDThreads) {
            const int gi = e / kC4, c4 = e % kC4;
            const float4* src = reinterpret_cast<const float4*>(pbase + (long long)gi * (D + 4) + 4) + c4;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 16
            for (int sp = 0; sp < n_splits; ++sp) {
                const float4 o = __ldcg(src + sp * sstride4);
                const float f = fws[sp * G + gi];
                acc.x = fmaf(o.x, f, acc.x);
                acc.y = fmaf(o.y, f, acc.y);
                acc.z = fmaf(o.z, f, acc.z);
                acc.w = fmaf(o.w, f, acc.w);
            }
            const float M = hml[2 * gi], L = hml[2 * gi + 1];
            const float inv = L > 0.0f ? 1.0f / L : 0.0f;
            const long long orow = (long long)b * Hq + (long long)h * G + gi;
            const float v[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
            if (out_f32) {
                reinterpret_cast<float4*>(static_cast<float*>(out) + orow * D)[c4] = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                T* dst = static_cast<T*>(out) + orow * D + 4 * c4;
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = from_f32<T>(v[k]);
            }
            if (lse && c4 == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    } else {
        for (int e = tid; e < G * D; e += kDThreads) {
            const int gi = e / D, ch = e % D;
            const float* base = pbase + (long long)gi * (D + 4);
            const long long sstride = (long long)G * (D + 4);
            float M = -INFINITY;
            for (int sp = 0; sp < n_splits; ++sp) {
                const float ls = __ldcg(base + sp * sstride + 1);
                if (ls > 0.0f) M = fmaxf(M, __ldcg(base + sp * sstride));
            }
            float L = 0.0f, O = 0.0f;
            for (int sp = 0; sp < n_splits; ++sp) {
                const float ls = __ldcg(base + sp * sstride + 1);
                if (ls > 0.0f) {
                    const float f = ex2(__ldcg(base + sp * sstride) - M);
                    L = fmaf(ls, f, L);
                    O = fmaf(__ldcg(base + sp * sstride + 4 + ch), f, O);
                }
            }
            const long long orow = (long long)b * Hq + (long long)h * G + gi;
            const float v = L > 0.0f ? O / L : 0.0f;
            if (out_f32) static_cast<float*>(out)[orow * D + ch] = v;
            else static_cast<T*>(out)[orow * D + ch] = from_f32<T>(v);
            if (lse && ch == 0) lse[orow] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
    }
}

// One CTA per stream, launched after the decode grid with programmatic stream
// serialisation: it may become resident while the decode grid runs, and waits for that grid
// to complete before reading.  CTA 0 also writes the call's status header from the decode
// CTAs' status words (word 0: the first wait code found, word 1: the range flag).
// Its shared memory is dynamic, and none up to 16 splits, so that its CTAs fit beside
// the decode CTAs still running on an SM and wait there.
template <typename T, int D>
__global__ void __launch_bounds__(kDThreads, 4) dec_merge_kernel(const float* __restrict__ part, int max_splits,
                                                                 int n_ctas, int Hkv, int B, int Hq,
                                                                 const int* __restrict__ cta_status,
                                                                 int* __restrict__ err, void* __restrict__ out,
                                                                 int out_f32, float* __restrict__ lse,
                                                                 int smem_floats) {
    extern __shared__ __align__(16) float msm[];
    __shared__ int s_code, s_range;
    const int tid = threadIdx.x;
    griddep_wait();
    if (blockIdx.x == 0) {
        if (tid == 0) s_code = s_range = 0;
        __syncthreads();
        for (int i = tid; i < n_ctas; i += kDThreads) {
            const int w = __ldcg(cta_status + i);
            if (w & 0xFFFF) atomicCAS(&s_code, 0, w & 0xFFFF);
            if (w >> 16) s_range = 1;
        }
        __syncthreads();
        if (tid == 0) {
            err[0] = s_code;
            err[1] = s_range;
        }
    }
    const int streams = B * Hkv, stream = blockIdx.x;
    const int n = n_ctas / streams + (stream < n_ctas % streams ? 1 : 0);
    if (n <= 1) return;
    const int G = Hq / Hkv;
    merge_splits<T, D>(part + (long long)stream * max_splits * G * (D + 4), n, G, stream / Hkv, stream % Hkv, Hq,
                       msm, smem_floats, out, out_f32, lse, tid);
}

// ------------------------------------------------------- operand dump -----
// Debug view of this kernel's own operands.  With fp32 metadata the kernel forms no
// dequantised key or value: the B/A operands of its quantised-block MMAs are the codes,
// turned into exact fp16 values by code_pair() with the lane constants above, and
// the steps and zeros enter through the query and probability sides; with fp16
// metadata the operands are the fp16 entries, one fp16x2 FMA of those codes with the
// (s, z) pairs.  This kernel runs that same extraction, per warp one block, on the
// block's words in global memory, and writes every fragment's fp16 values at their
// (token, channel) place: Kout/Vout fp16 [B][Hkv][32 n_total][d] in stream slot order
// (all segments' blocks in memory order).  RAW16 slots are not written (they enter as
// stored).
template <int D, int BITS>
__global__ void __launch_bounds__(32)
dec_operands_kernel(DevCache c, int seg, int slot0, int n_total, __half* __restrict__ Kout,
                    __half* __restrict__ Vout) {
    const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x;
    const LaneConst lc = lane_const(lane);
    const unsigned char* blk = block_ptr(c, b, h, seg, i);
    const IntBlockOffsets o = int_offsets(D, BITS, c.meta16);
    const long long base = (((long long)b * c.Hkv + h) * n_total + slot0 + i) * kBlockTokens;
    auto put = [&](__half* out, int tok, int ch, uint32_t pair) {
        *reinterpret_cast<uint32_t*>(out + (base + tok) * D + ch) = pair;
    };
    auto put_t = [&](__half* out, int ch, int tok, uint32_t pair) {   // pair = (tok, tok + 1) of channel ch
        const __half2 v = *reinterpret_cast<const __half2*>(&pair);
        out[(base + tok) * D + ch] = __low2half(v);
        out[(base + tok + 1) * D + ch] = __high2half(v);
    };
    constexpr int KW = D * BITS / 32;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk + o.kc);
#pragma unroll 1
    for (int mt = 0; mt < 2; ++mt) {
        const int ka = 16 * mt + lc.g, kb = ka + 8;
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c0 = 16 * kk + 2 * lc.tig;
            uint32_t a[4];
            if (BITS == 2) {
                const uint32_t wa = kc[ka * KW + kk], wb = kc[kb * KW + kk];
                a[0] = code_pair(wa, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[1] = code_pair(wb, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[2] = code_pair(wa, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                a[3] = code_pair(wb, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                a[0] = code_pair(kc[ka * KW + 2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[1] = code_pair(kc[kb * KW + 2 * kk], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[2] = code_pair(kc[ka * KW + 2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[3] = code_pair(kc[kb * KW + 2 * kk + 1], lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
            if (c.meta16) {   // fp16 metadata: the kernel's operands are the entries themselves
                const uint32_t* km = reinterpret_cast<const uint32_t*>(blk + o.km);
                const uint2 m0 = *reinterpret_cast<const uint2*>(km + c0);
                const uint2 m1 = *reinterpret_cast<const uint2*>(km + c0 + 8);
                a[0] = hfma2_u32(a[0], __byte_perm(m0.x, m0.y, 0x5410), __byte_perm(m0.x, m0.y, 0x7632));
                a[1] = hfma2_u32(a[1], __byte_perm(m0.x, m0.y, 0x5410), __byte_perm(m0.x, m0.y, 0x7632));
                a[2] = hfma2_u32(a[2], __byte_perm(m1.x, m1.y, 0x5410), __byte_perm(m1.x, m1.y, 0x7632));
                a[3] = hfma2_u32(a[3], __byte_perm(m1.x, m1.y, 0x5410), __byte_perm(m1.x, m1.y, 0x7632));
            }
            // m16n8k16 A fragment: rows (keys) g, g + 8; columns (channels) 2 tig, 2 tig + 8
            put(Kout, ka, c0, a[0]);
            put(Kout, kb, c0, a[1]);
            put(Kout, ka, c0 + 8, a[2]);
            put(Kout, kb, c0 + 8, a[3]);
        }
    }
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + o.vc);
#pragma unroll 1
    for (int cm = 0; cm < D / 16; ++cm) {
        const int ca = 16 * cm + lc.g, cb = ca + 8;
#pragma unroll 1
        for (int kk = 0; kk < 2; ++kk) {
            const int t0 = 16 * kk + 2 * lc.tig;
            uint32_t a[4];
            if (BITS == 2) {
                const uint32_t wa = vc[ca * 2 + kk], wb = vc[cb * 2 + kk];
                a[0] = code_pair(wa, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[1] = code_pair(wb, lc.sel2a, lc.mask2, lc.scale2, lc.bias2);
                a[2] = code_pair(wa, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
                a[3] = code_pair(wb, lc.sel2b, lc.mask2, lc.scale2, lc.bias2);
            } else {
                const uint2 wa = *reinterpret_cast<const uint2*>(vc + ca * 4 + 2 * kk);
                const uint2 wb = *reinterpret_cast<const uint2*>(vc + cb * 4 + 2 * kk);
                a[0] = code_pair(wa.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[1] = code_pair(wb.x, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[2] = code_pair(wa.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
                a[3] = code_pair(wb.y, lc.sel4, 0x00F0000Fu, lc.scale4, lc.bias4);
            }
            if (c.meta16) {
                const uint32_t* vm = reinterpret_cast<const uint32_t*>(blk + o.vm) + (cm >> 1) * 32;
                const uint2 m0 = *reinterpret_cast<const uint2*>(vm + t0);
                const uint2 m1 = *reinterpret_cast<const uint2*>(vm + t0 + 8);
                a[0] = hfma2_u32(a[0], __byte_perm(m0.x, m0.y, 0x5410), __byte_perm(m0.x, m0.y, 0x7632));
                a[1] = hfma2_u32(a[1], __byte_perm(m0.x, m0.y, 0x5410), __byte_perm(m0.x, m0.y, 0x7632));
                a[2] = hfma2_u32(a[2], __byte_perm(m1.x, m1.y, 0x5410), __byte_perm(m1.x, m1.y, 0x7632));
                a[3] = hfma2_u32(a[3], __byte_perm(m1.x, m1.y, 0x5410), __byte_perm(m1.x, m1.y, 0x7632));
            }
            // rows (channels) g, g + 8; columns (tokens) 2 tig, 2 tig + 8
            put_t(Vout, ca, t0, a[0]);
            put_t(Vout, cb, t0, a[1]);
            put_t(Vout, ca, t0 + 8, a[2]);
            put_t(Vout, cb, t0 + 8, a[3]);
        }
    }
}

template <int D>
kv_status launch_dec_operands_d(const DevCache& c, void* Kout, void* Vout, cudaStream_t st) {
    const int n_total = c.n_blocks[0] + c.n_blocks[1] + c.n_blocks[2];
    int slot0 = 0;
    for (int seg = 0; seg < KV_NUM_SEG; ++seg) {
        const int cls = seg_class(c.kind, seg), nb = c.n_blocks[seg];
        if (nb > 0 && (cls == CLS_INT2 || cls == CLS_INT4)) {
            const dim3 grid(nb, c.Hkv, c.B);
            if (cls == CLS_INT2)
                dec_operands_kernel<D, 2><<<grid, 32, 0, st>>>(c, seg, slot0, n_total, static_cast<__half*>(Kout),
                                                               static_cast<__half*>(Vout));
            else
                dec_operands_kernel<D, 4><<<grid, 32, 0, st>>>(c, seg, slot0, n_total, static_cast<__half*>(Kout),
                                                               static_cast<__half*>(Vout));
            const kv_status s = check_launch("dec_operands_kernel");
            if (s != KV_OK) return s;
        }
        slot0 += nb;
    }
    return KV_OK;
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
    sh.rows = Hq / L.Hkv > 8 ? 16 : 8;   // heads per warp row block: 8 NT
    return sh;
}

size_t dec_smem_bytes(const DecShape& sh, int d) {
    return 1024 + (size_t)kDW * sh.nsw * sh.slot_bytes + (size_t)kDW * sh.rows * (d + 2) * sizeof(float) +
           (size_t)kDW * sh.nsw * 8 + 8;
}

// One status word per decode CTA (at most n_splits per stream), in 256-byte units.
size_t dec_status_bytes(const kv_cache* cache, int n_splits) {
    return ((size_t)cache->layout.B * cache->layout.Hkv * n_splits * sizeof(int) + 255) / 256 * 256;
}

template <typename T, int D, int NT, int JENSEN, bool M16>
kv_status launch_dec_t(const void* Q, const void* Kc, const void* Vc, int n_cur, int Hq, const kv_cache* cache,
                       float tau, int n_splits, int n_ctas, void* out, int out_f32, float* lse, void* ws,
                       cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    const DecShape sh = dec_shape(cache, Hq);
    const size_t smem = dec_smem_bytes(sh, D);
    const kv_status sa = set_smem_limit(reinterpret_cast<const void*>(attn_decode_kernel<T, D, NT, JENSEN, M16>), smem,
                                        "attn_decode_kernel");
    if (sa != KV_OK) return sa;
    unsigned char* w = static_cast<unsigned char*>(ws);
    int* err = reinterpret_cast<int*>(w);
    int* cta_status = reinterpret_cast<int*>(w + kStatusBytes);
    float* part = reinterpret_cast<float*>(w + kStatusBytes + dec_status_bytes(cache, n_splits));
    // n_ctas CTAs over the B * Hkv streams, at most n_splits per stream (0: n_splits each)
    const int streams = c.B * c.Hkv;
    if (n_ctas <= 0 || n_ctas > streams * n_splits) n_ctas = streams * n_splits;
    if (n_ctas < streams) n_ctas = streams;
    attn_decode_kernel<T, D, NT, JENSEN, M16><<<n_ctas, kDThreads, smem, st>>>(
        static_cast<const T*>(Q), static_cast<const T*>(Kc), static_cast<const T*>(Vc), n_cur, Hq, c, tau, n_splits,
        n_ctas, sh, out, out_f32, lse, part, cta_status, getenv("BITKV_TEST_NEVER_ARRIVE") != nullptr ? 1 : 0);
    const kv_status sk = check_launch("attn_decode_kernel");
    if (sk != KV_OK) return sk;
    // the merge grid (and the status header) follows with programmatic stream serialisation
    const int G = Hq / c.Hkv;
    int mfloats = 0;
    if (n_splits > 16) mfloats = 3 * n_splits * G + 2 * G < kMergeSmemFloats ? 3 * n_splits * G + 2 * G : 0;
    static bool carveout_set = false;
    if (!carveout_set) {
        // the decode kernel runs at the largest shared-memory carveout; the same for the
        // merge kernel lets its CTAs share an SM with decode CTAs
        for (auto* k : {dec_merge_kernel<__half, 64>, dec_merge_kernel<__half, 128>,
                        dec_merge_kernel<__nv_bfloat16, 64>, dec_merge_kernel<__nv_bfloat16, 128>})
            cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        carveout_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(streams);
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = (size_t)mfloats * sizeof(float);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* cpart = part;
    const int* cstat = cta_status;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, dec_merge_kernel<T, D>, cpart, n_splits, n_ctas, c.Hkv, c.B, Hq,
                                             cstat, err, out, out_f32, lse, mfloats);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "dec_merge_kernel launch: %s", cudaGetErrorString(e));
    return check_launch("dec_merge_kernel");
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

// Resident CTAs of the decode kernel on the whole GPU (shared memory bounds them).
int decode_resident_ctas(const kv_cache* cache, int Hq) {
    const DecShape sh = dec_shape(cache, Hq);
    const size_t smem = dec_smem_bytes(sh, cache->layout.d);
    int per_sm = (int)((228 * 1024) / (smem + 1024));
    if (per_sm > 16) per_sm = 16;
    if (per_sm < 1) per_sm = 1;
    return per_sm * dec_num_sms();
}

// Automatic split count: the most splits any stream takes when one wave of resident
// CTAs is spread over the streams (some streams then take one split fewer; see
// decode_auto_ctas), with at least two blocks per warp.
int decode_auto_splits(const kv_cache* cache, int Hq) {
    const kv_layout& L = cache->layout;
    const int streams = L.B * L.Hkv > 0 ? L.B * L.Hkv : 1;
    const int nb = cache->n_blocks[0] + cache->n_blocks[1] + cache->n_blocks[2];
    const int slots = decode_resident_ctas(cache, Hq);
    int s = (slots + streams - 1) / streams;
    const int cap = nb / (2 * kDW) > 1 ? nb / (2 * kDW) : 1;   // at least two blocks per warp
    if (s > cap) s = cap;
    return s < 1 ? 1 : s;
}

// Automatic CTA count: one full wave of resident CTAs (never more than n_splits per
// stream, never fewer than one per stream).
int decode_auto_ctas(const kv_cache* cache, int Hq, int n_splits) {
    const kv_layout& L = cache->layout;
    const int streams = L.B * L.Hkv;
    const int slots = decode_resident_ctas(cache, Hq);
    int n = slots < streams * n_splits ? slots : streams * n_splits;
    return n < streams ? streams : n;
}

size_t decode_workspace(const kv_cache* cache, int Hq, int n_splits) {
    const kv_layout& L = cache->layout;
    const int G = Hq / L.Hkv;
    size_t ws = kStatusBytes + dec_status_bytes(cache, n_splits);
    if (n_splits > 1) ws += (size_t)L.B * L.Hkv * n_splits * G * (L.d + 4) * sizeof(float);
    return ws;
}

kv_status launch_attn_decode(const void* Q, const void* Kc, const void* Vc, kv_dtype dt, int n_cur, int Hq,
                             const kv_cache* cache, float tau, int jensen, int n_splits, int n_ctas, void* out,
                             int out_f32, float* lse, void* ws, cudaStream_t st) {
    const int d = cache->layout.d;
    const bool two = Hq / cache->layout.Hkv > 8;
    const bool m16 = cache->layout.meta_dtype == KV_F16;
    using F16 = __half;
    using BF16 = __nv_bfloat16;
#define BITKV_DEC_M(T, D, NT, M16)                                                                             \
    do {                                                                                                        \
        if (jensen == KV_JENSEN_TAYLOR2)                                                                        \
            return launch_dec_t<T, D, NT, KV_JENSEN_TAYLOR2, M16>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits, \
                                                                   n_ctas, out, out_f32, lse, ws, st);                  \
        if (jensen == KV_JENSEN_EXACT)                                                                          \
            return launch_dec_t<T, D, NT, KV_JENSEN_EXACT, M16>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits,   \
                                                                 n_ctas, out, out_f32, lse, ws, st);                    \
        if (jensen == KV_JENSEN_ISOTROPIC)                                                                      \
            return launch_dec_t<T, D, NT, KV_JENSEN_ISOTROPIC, M16>(Q, Kc, Vc, n_cur, Hq, cache, tau,         \
                                                                     n_splits, n_ctas, out, out_f32, lse, ws, st);      \
        return launch_dec_t<T, D, NT, KV_JENSEN_OFF, M16>(Q, Kc, Vc, n_cur, Hq, cache, tau, n_splits, n_ctas, \
                                                           out, out_f32, lse, ws, st);                               \
    } while (0)
#define BITKV_DEC(T, D, NT)                                                                                    \
    do {                                                                                                        \
        if (m16) BITKV_DEC_M(T, D, NT, true);                                                                   \
        BITKV_DEC_M(T, D, NT, false);                                                                           \
    } while (0)
    if (dt == KV_F16) {
        if (d == 64) { if (two) BITKV_DEC(F16, 64, 2); else BITKV_DEC(F16, 64, 1); }
        else { if (two) BITKV_DEC(F16, 128, 2); else BITKV_DEC(F16, 128, 1); }
    } else {
        if (d == 64) { if (two) BITKV_DEC(BF16, 64, 2); else BITKV_DEC(BF16, 64, 1); }
        else { if (two) BITKV_DEC(BF16, 128, 2); else BITKV_DEC(BF16, 128, 1); }
    }
#undef BITKV_DEC
#undef BITKV_DEC_M
}

kv_status launch_dec_operands(const kv_cache* cache, void* Kout, void* Vout, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    if (c.kind == KV_CODEBOOK2) return set_error(KV_ERR_UNSUPPORTED, "decode operands: codebook caches not served");
    if (c.d == 64) return launch_dec_operands_d<64>(c, Kout, Vout, st);
    if (c.d == 128) return launch_dec_operands_d<128>(c, Kout, Vout, st);
    return set_error(KV_ERR_UNSUPPORTED, "decode operands: needs head dim 64 or 128");
}

}  // namespace bitkv
