// Shared device/host definitions of libbitkv: block format, dtype helpers,
// and the dequantisation routine every kernel uses.
//
// Block format (32 token slots of one batch row and kv head), head dim d:
//   INT2/INT4 (b bits): Kc u32[32][d*b/32] token-major | Km float2[d] |
//                       Vc u32[d][b] channel-major     | Vm float2[d/32][32]
//   RAW16:              K 16-bit[32][d] | V 16-bit[32][d], 16-byte chunk j of row t
//                       stored at chunk position j ^ (t mod min(8, d/8))
//   CODEBOOK2:          Kc u32[32][d/16] | Vc u32[d][2] | Vm float2[d/32][32] | Kq fp16[32][rp]
// fp16-metadata layouts store Km as half2[d] and Vm as half2[d/32][32] (INT blocks only).
// Quantiser (step sizes of "Quantized Keys Steal Attention", abstract; INT2/INT4
// of the WindowQuant note, table in 何が新しいのか):
//   s = fl32(fl32(M-m)/(2^b-1)), code = clamp(rint(fl32(fl32(x-m)/s))), z = m,
//   x_hat = fmaf(code, s, z).
// With fp16 metadata s and z are first rounded to fp16 (a -0 zero point as +0), the
// codes are taken against the rounded pair, and x_hat = fp16(code * s + z) with one
// rounding (an fp16 FMA).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/bitkv.h"

namespace bitkv {

constexpr int kBlockTokens = 32;

// Everything a kernel needs to address a cache, passed by value.
struct DevCache {
    unsigned char* data;
    int32_t* blk_len;
    int32_t* blk_pos;
    const float* centroids;
    const float* psac_u;
    const float* resid_var;        // CODEBOOK2 residual variances [B][Hkv][d], or NULL
    int B, Hkv, d, kind, raw_dtype, r, rp;
    int meta16;                    // INT blocks store (s, z) as fp16 pairs
    int cap_total;
    int seg_base[KV_NUM_SEG];      // index of a segment's first block in blk_len / blk_pos rows
    int n_blocks[KV_NUM_SEG];
    long long block_bytes[KV_NUM_SEG];
    long long seg_offset[KV_NUM_SEG];
    long long stream_bytes;
};

// Segment class of segment k for a cache kind: 16, 4 or 2 bits, or 3 for codebook.
enum SegClass { CLS_RAW16 = 0, CLS_INT4 = 1, CLS_INT2 = 2, CLS_CB2 = 3 };

__host__ __device__ inline int seg_class(int kind, int seg) {
    if (kind == KV_CODEBOOK2) return CLS_CB2;
    return seg;  // RAW16 / INT4 / INT2 by segment position
}

__host__ __device__ inline unsigned char* block_ptr(const DevCache& c, int b, int h, int seg, int i) {
    return c.data + ((long long)b * c.Hkv + h) * c.stream_bytes + c.seg_offset[seg] +
           (long long)i * c.block_bytes[seg];
}

// Byte offsets of the sub-arrays inside a block.
struct IntBlockOffsets {
    int kc, km, vc, vm;
};
__host__ __device__ inline IntBlockOffsets int_offsets(int d, int bits, int meta16) {
    IntBlockOffsets o;
    o.kc = 0;
    o.km = 4 * d * bits;
    o.vc = o.km + (meta16 ? 4 : 8) * d;
    o.vm = o.vc + 4 * d * bits;
    return o;
}

// (s, z) pair i of a metadata array: fp32 pairs, or fp16 pairs widened exactly.
template <bool M16>
__device__ __forceinline__ float2 meta_at(const unsigned char* base, int i) {
    if constexpr (M16) return __half22float2(reinterpret_cast<const __half2*>(base)[i]);
    else return reinterpret_cast<const float2*>(base)[i];
}
__device__ __forceinline__ float2 meta_at(const unsigned char* base, int i, int meta16) {
    return meta16 ? meta_at<true>(base, i) : meta_at<false>(base, i);
}
// Pairs i and i + 1 (i even) as (s_i, z_i, s_i+1, z_i+1), one 16- or 8-byte load.
template <bool M16>
__device__ __forceinline__ float4 meta2_at(const unsigned char* base, int i) {
    if constexpr (M16) {
        const uint2 u = reinterpret_cast<const uint2*>(base)[i >> 1];
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    } else {
        return reinterpret_cast<const float4*>(base)[i >> 1];
    }
}
struct CbBlockOffsets {
    int kc, vc, vm, kq;
};
__host__ __device__ inline CbBlockOffsets cb_offsets(int d) {
    CbBlockOffsets o;
    o.kc = 0;
    o.vc = 8 * d;
    o.vm = 16 * d;
    o.kq = 24 * d;
    return o;
}

// The one dequantisation rule: one fp32 rounding of code*s + z.
__device__ __forceinline__ float dequant(uint32_t code, float s, float z) {
    return __fmaf_rn(__uint2float_rn(code), s, z);
}

// fp16 dequantisation of blocks with fp16 metadata: one rounding of code * s + z, where
// sz holds (s, z) as an fp16 pair; the code (< 16) is exact in fp16.
__device__ __forceinline__ float dequant_h(uint32_t code, __half2 sz) {
    return __half2float(__hfma(__uint2half_rn(code), __low2half(sz), __high2half(sz)));
}

// Codes i and i + 1 (i even) of a b-bit packed word as an exact fp16 pair (code i in the
// low half).  The byte holding both codes goes into both halves, a mask keeps code i in
// the low half and code i + 1 (times 2^b) in the high half, the fp16 exponent of 1024 is
// or-ed in (values 1024 + code 2^p), and one fp16x2 FMA takes off the 1024 and the 2^p;
// every step is exact.  With i known at compile time the constants fold.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t w, int i) {
    const uint32_t byte = BITS == 2 ? (uint32_t)(i >> 2) : (uint32_t)(i >> 1);
    const uint32_t sel = byte | 0x40u | (byte << 8) | 0x4000u;
    uint32_t mask, scale, bias;
    if (BITS == 2) {
        const bool hi = (i >> 1) & 1;      // codes in bits 4-7 of the byte
        mask = hi ? 0x00C00030u : 0x000C0003u;
        scale = hi ? 0x24002C00u : 0x34003C00u;   // (2^-4, 2^-6) : (1, 2^-2)
        bias = hi ? 0xCC00D400u : 0xDC00E400u;    // (-64, -16) : (-1024, -256)
    } else {
        mask = 0x00F0000Fu;
        scale = 0x2C003C00u;                      // (1, 2^-4)
        bias = 0xD400E400u;                       // (-1024, -64)
    }
    const uint32_t x = (__byte_perm(w, 0u, sel) & mask) | 0x64006400u;
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(scale), "r"(bias));
    return r;
}

// fp16x2 FMA a * b + c, one rounding per half.
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Key code of (token t, channel c) in a token-major code array.
__device__ __forceinline__ uint32_t key_code(const uint32_t* kc, int t, int c, int d, int bits) {
    const int per = 32 / bits;
    const uint32_t w = kc[t * (d / per) + c / per];
    return (w >> (bits * (c % per))) & ((1u << bits) - 1u);
}
// Value code of (token t, channel c) in a channel-major code array.
__device__ __forceinline__ uint32_t val_code(const uint32_t* vc, int t, int c, int bits) {
    const int per = 32 / bits;
    const uint32_t w = vc[c * bits + t / per];
    return (w >> (bits * (t % per))) & ((1u << bits) - 1u);
}

// 16-bit slot of element (t, c) inside the K (or V) half of a RAW16 block: the
// row's 16-byte chunks are XOR-permuted by the token index so that eight
// consecutive rows of one chunk column occupy distinct shared-memory banks.
__host__ __device__ __forceinline__ int raw16_slot(int t, int c, int d) {
    const int m = (d >= 64 ? 8 : d / 8) - 1;
    return t * d + ((((c >> 3) ^ (t & m))) << 3) + (c & 7);
}

// ---- dtype helpers ---------------------------------------------------------
__device__ __forceinline__ float raw16_to_f32(uint16_t bits, int raw_dtype);

// Dequantised (key, value) of token t, channel ch of one block, in fp32 before
// any rounding to the I/O dtype.  `cent` is the [d][4] centroid table of the
// block's (batch, kv head) for codebook blocks, else unused.
__device__ __forceinline__ float2 block_entry(int cls, const unsigned char* blk, int d, int raw_dtype, int meta16,
                                              const float* cent, int t, int ch) {
    if (cls == CLS_RAW16) {
        const uint16_t* r = reinterpret_cast<const uint16_t*>(blk);
        const int slot = raw16_slot(t, ch, d);
        return make_float2(raw16_to_f32(r[slot], raw_dtype), raw16_to_f32(r[kBlockTokens * d + slot], raw_dtype));
    }
    if (cls == CLS_CB2) {
        const CbBlockOffsets o = cb_offsets(d);
        const uint32_t ki = key_code(reinterpret_cast<const uint32_t*>(blk + o.kc), t, ch, d, 2);
        const float2 sv = reinterpret_cast<const float2*>(blk + o.vm)[(ch / 32) * 32 + t];
        const uint32_t vq = val_code(reinterpret_cast<const uint32_t*>(blk + o.vc), t, ch, 2);
        return make_float2(cent[ch * 4 + ki], dequant(vq, sv.x, sv.y));
    }
    const int bits = cls == CLS_INT4 ? 4 : 2;
    const IntBlockOffsets o = int_offsets(d, bits, meta16);
    const uint32_t kq = key_code(reinterpret_cast<const uint32_t*>(blk + o.kc), t, ch, d, bits);
    const uint32_t vq = val_code(reinterpret_cast<const uint32_t*>(blk + o.vc), t, ch, bits);
    if (meta16)
        return make_float2(dequant_h(kq, reinterpret_cast<const __half2*>(blk + o.km)[ch]),
                           dequant_h(vq, reinterpret_cast<const __half2*>(blk + o.vm)[(ch / 32) * 32 + t]));
    const float2 sk = meta_at<false>(blk + o.km, ch);
    const float2 sv = meta_at<false>(blk + o.vm, (ch / 32) * 32 + t);
    return make_float2(dequant(kq, sk.x, sk.y), dequant(vq, sv.x, sv.y));
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Raw 16-bit cache entry to fp32.
__device__ __forceinline__ float raw16_to_f32(uint16_t bits, int raw_dtype) {
    if (raw_dtype == KV_BF16) return __uint_as_float(((uint32_t)bits) << 16);
    return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// log(sinh(x)/x): the Taylor series of the log (Bernoulli-number
// coefficients 1/6, -1/180, 1/2835, -1/37800) below 0.5, where its truncation
// error is < 1e-8; above, x + log(1 - exp(-2x)) - log(2x) with the fast
// hardware exp and log: there 1 - exp(-2x) >= 0.63 and 2x >= 1, so nothing
// cancels and the absolute error stays near 1e-6.
__device__ __forceinline__ float log_sinhc_series(float x) {
    const float x2 = x * x;
    return x2 * (1.0f / 6.0f + x2 * (-1.0f / 180.0f + x2 * (1.0f / 2835.0f - x2 * (1.0f / 37800.0f))));
}
__device__ __forceinline__ float log_sinhc(float x) {
    x = fabsf(x);
    if (x < 0.5f) return log_sinhc_series(x);
    return x + __logf(1.0f - __expf(-2.0f * x)) - __logf(2.0f * x);
}

// Every attention workspace starts with a status header of kStatusBytes: int word 0
// holds the code of a bounded device-side wait that gave up (0: none), word 1 the
// range flag (an fp16 operand of the tensor-core path would be infinite).  The
// tensor-core and CUDA-core calls clear the header before their kernels run; the
// decode call's merge kernel writes it.
constexpr size_t kStatusBytes = 256;

// Host-side helpers shared by the launch code.
DevCache make_dev_cache(const kv_cache* c);
// Zeroes `bytes` of device memory at `p` on `st` (the status header and whatever
// else a launch needs cleared); KV_ERR_CUDA if the runtime refuses.
kv_status clear_device(void* p, size_t bytes, cudaStream_t st, const char* who);
// Copies the status header at `ws` to the host after the work queued on `st` and
// maps it to KV_OK, KV_ERR_TIMEOUT or KV_ERR_RANGE.  Synchronises `st`.
kv_status read_status(const void* ws, cudaStream_t st);
kv_status set_error(kv_status st, const char* fmt, ...);
kv_status check_launch(const char* what);
// An NVTX range named for a C-ABI call, open for the call's duration: a profiler
// (nsys, ncu's range filters) then shows each call with the kernels it launched.
// Without an attached tool the push and pop do nothing.
struct AbiRange {
    explicit AbiRange(const char* name) { nvtxRangePushA(name); }
    ~AbiRange() { nvtxRangePop(); }
    AbiRange(const AbiRange&) = delete;
    AbiRange& operator=(const AbiRange&) = delete;
};

// Raises `kernel`'s dynamic shared-memory limit on the current device to at least
// `bytes`, once per (kernel, device), never lowering it; thread-safe.  KV_ERR_CUDA
// (with the message set) when the runtime refuses.
kv_status set_smem_limit(const void* kernel, size_t bytes, const char* name);

}  // namespace bitkv
