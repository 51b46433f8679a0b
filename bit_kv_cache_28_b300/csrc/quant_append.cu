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

__device__ __forceinline__ uint32_t code_of(float x, float s, float z, float qmax) {
    if (!(s > 0.0f)) return 0u;
    float t = rintf(__fdiv_rn(__fsub_rn(x, z), s));  // ties to even
    t = fminf(fmaxf(t, 0.0f), qmax);
    return static_cast<uint32_t>(t);
}

// Values of one block: per (token, 32-channel group) with a warp per group.
// Writes Vm[g][t] and the value codes into codes[t][ch].
template <int BITS>
__device__ void quantise_values(const float* Vs, int ld, int d, int nv, uint8_t* codes, float2* vm) {
    const float qmax = float((1 << BITS) - 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int ng = d / 32;
    for (int p = warp; p < kBlockTokens * ng; p += nwarps) {
        const int t = p / ng, g = p % ng;
        const float x = Vs[t * ld + g * 32 + lane];
        float s = 0.0f, z = 0.0f;
        uint32_t q = 0;
        if (t < nv) {                                  // warp-uniform
            const float mn = warp_min(x), mx = warp_max(x);
            step_and_zero(mn, mx, qmax, s, z);
            q = code_of(x, s, z, qmax);
        }
        codes[t * d + g * 32 + lane] = static_cast<uint8_t>(q);
        if (lane == 0) vm[g * 32 + t] = make_float2(s, z);
    }
}

// Pack codes[t][ch] channel-major: word (ch, q) holds tokens q*per .. q*per+per-1.
template <int BITS>
__device__ void pack_values(const uint8_t* codes, int d, uint32_t* vcw) {
    constexpr int per = 32 / BITS;
    for (int w = threadIdx.x; w < d * BITS; w += blockDim.x) {
        const int ch = w / BITS, q = w % BITS;
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) v |= uint32_t(codes[(q * per + i) * d + ch]) << (BITS * i);
        vcw[w] = v;
    }
}

// Pack codes[t][ch] token-major: word (t, q) holds channels q*per .. q*per+per-1.
template <int BITS>
__device__ void pack_keys(const uint8_t* codes, int d, uint32_t* kcw) {
    constexpr int per = 32 / BITS;
    const int wpr = d / per;
    for (int w = threadIdx.x; w < kBlockTokens * wpr; w += blockDim.x) {
        const int t = w / wpr, q = w % wpr;
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) v |= uint32_t(codes[t * d + q * per + i]) << (BITS * i);
        kcw[w] = v;
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

// One uniform INT block.  Keys: channel c is shared by tpc = 256 / d adjacent
// threads, each taking 32 / tpc tokens; min / max are combined by shuffles.
// Values: (token t, 32-channel group g) is shared by tpc threads the same way.
// Codes go to byte arrays kc8[t][c] and vc8[c][t]; one thread per output word
// packs them.
template <int BITS>
__device__ void encode_int_block(const float* Ks, const float* Vs, int ld, int d, int nv, uint8_t* kc8,
                                 uint8_t* vc8, unsigned char* blk) {
    const float qmax = float((1 << BITS) - 1);
    const IntBlockOffsets o = int_offsets(d, BITS);
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
        const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
        if (part == 0) reinterpret_cast<float2*>(blk + o.km)[ch] = make_float2(s, z);
        for (int i = 0; i < span; ++i) {
            const int t = t0 + i;
            kc8[t * d + ch] = t < nv ? static_cast<uint8_t>(code_fast(Ks[t * ld + ch], s, r, z, qmax)) : 0;
        }
    }
    // values: per (token, 32-channel group); pair index = t * (d / 32) + g
    {
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
        const float r = s > 0.0f ? __frcp_rn(s) : 0.0f;
        if (part == 0) reinterpret_cast<float2*>(blk + o.vm)[g * 32 + t] = make_float2(s, z);
        for (int i = 0; i < span; ++i)
            vc8[(c0 + i) * kBlockTokens + t] =
                t < nv ? static_cast<uint8_t>(code_fast(Vs[t * ld + c0 + i], s, r, z, qmax)) : 0;
    }
    __syncthreads();
    // pack: key word (t, q) holds channels q per .. q per + per - 1 of token t;
    // value word (c, q) holds tokens q per .. of channel c (per = 32 / BITS)
    constexpr int per = 32 / BITS;
    uint32_t* kw = reinterpret_cast<uint32_t*>(blk + o.kc);
    uint32_t* vw = reinterpret_cast<uint32_t*>(blk + o.vc);
    const int nwords = kBlockTokens * d / per;    // same count for keys and values
    for (int w = tid; w < nwords; w += kAppendThreads) {
        const uint8_t* ksrc = kc8 + w * per;        // token-major bytes: word w covers bytes w per ..
        const uint8_t* vsrc = vc8 + w * per;        // channel-major bytes, likewise
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

// Codebook block: nearest fp32 centroid per key entry (fp64 |x - mu|, ties to
// the lower index), INT2 values, fp16 PSAC coefficients U^T (k - k_hat) in fp64.
__device__ void encode_cb_block(const float* Ks, const float* Vs, int ld, int d, int nv, uint8_t* codes,
                                unsigned char* blk, const float* cent, const float* U, int r, int rp) {
    const CbBlockOffsets o = cb_offsets(d);
    for (int ch = threadIdx.x; ch < d; ch += blockDim.x) {
        const double mu0 = cent[ch * 4 + 0], mu1 = cent[ch * 4 + 1], mu2 = cent[ch * 4 + 2], mu3 = cent[ch * 4 + 3];
        for (int t = 0; t < kBlockTokens; ++t) {
            uint8_t k = 0;
            if (t < nv) {
                const double x = Ks[t * ld + ch];
                double best = fabs(x - mu0);
                const double d1 = fabs(x - mu1), d2 = fabs(x - mu2), d3 = fabs(x - mu3);
                if (d1 < best) { best = d1; k = 1; }
                if (d2 < best) { best = d2; k = 2; }
                if (d3 < best) { best = d3; k = 3; }
            }
            codes[t * d + ch] = k;
        }
    }
    __syncthreads();
    pack_keys<2>(codes, d, reinterpret_cast<uint32_t*>(blk + o.kc));
    // PSAC coefficients before the scratch is reused for values
    __half* kq = reinterpret_cast<__half*>(blk + o.kq);
    for (int e = threadIdx.x; e < kBlockTokens * rp; e += blockDim.x) {
        const int t = e / rp, j = e % rp;
        double acc = 0.0;
        if (t < nv && j < r) {
            for (int ch = 0; ch < d; ++ch) {
                const double khat = cent[ch * 4 + codes[t * d + ch]];
                acc += (double)U[ch * r + j] * ((double)Ks[t * ld + ch] - khat);
            }
        }
        kq[e] = __double2half(acc);
    }
    __syncthreads();
    quantise_values<2>(Vs, ld, d, nv, codes, reinterpret_cast<float2*>(blk + o.vm));
    __syncthreads();
    pack_values<2>(codes, d, reinterpret_cast<uint32_t*>(blk + o.vc));
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
            encode_int_block<4>(Ks, Vs, ld, d, nv, codes, codes + kBlockTokens * d, blk);
        } else if (cls == CLS_INT2) {
            encode_int_block<2>(Ks, Vs, ld, d, nv, codes, codes + kBlockTokens * d, blk);
        } else {
            const long long bh = (long long)b * c.Hkv + h;
            encode_cb_block(Ks, Vs, ld, d, nv, codes, blk, c.centroids + bh * d * 4,
                            c.r > 0 ? c.psac_u + bh * d * c.r : nullptr, c.r, c.rp);
        }
    }
    if (h == 0 && threadIdx.x == 0) {
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
        const float2 kv = block_entry(cls, blk, d, c.raw_dtype, cent, t, ch);
        const long long o = (((long long)b * c.Hkv + h) * n_tok + pos + t) * d + ch;
        Kout[o] = kv.x;
        Vout[o] = kv.y;
    }
}

}  // namespace

size_t append_smem_bytes(int d) {
    return 2 * kBlockTokens * (d + 1) * sizeof(float) + 2 * kBlockTokens * d;
}

template <typename T>
static kv_status launch_append_t(const void* K, const void* V, int n_tokens, const kv_cache* cache, int mode,
                                 int uni_seg, const int8_t* win_bits, int n_win, int grid_x, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    const size_t sm = append_smem_bytes(c.d);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(append_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
        attr_set = true;
    }
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
