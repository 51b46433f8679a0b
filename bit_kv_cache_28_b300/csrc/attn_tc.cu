// Tensor-core (tcgen05 / TMEM) attention of a chunk of queries over a packed
// INT2 / INT4 cache plus the current, unquantised chunk, bf16 I/O, head dim 128.
//
// "Quantized Keys Steal Attention" (abstract): chunk-wise autoregressive
// attention over an INT2 cache with a per-score Jensen correction computed on
// the fly from the cached keys' step sizes and the query (second-order form:
// delta = tau^2/24 sum_c q_c^2 s_c^2).  The dequantisation never leaves the SM
// (the self-forcing KV study's lesson that rebuilding full bf16 buffers defeats
// the compression): packed blocks are expanded into shared-memory operand tiles.
//
// One CTA = 128 queries of one (batch, head) x a range of 128-key tiles.
//   warps 0-3   softmax: thread i owns query row i = TMEM lane i.  Two passes
//               over the S row in TMEM (row maximum per 32-key group, then
//               p = 2^(S c1 - (m + delta_g))), a lazily rescaled running max (O is
//               rescaled only when the max grows by more than 2^15), P written
//               back to TMEM as fp16.
//   warps 4-11  producers: thread 0 bulk-copies (TMA engine) each packed cache
//               tile -- 4 contiguous blocks -- into a double-buffered staging
//               area two tiles ahead; all 256 threads expand the staged codes
//               into K_hat [128 keys x 128] (fp16, single buffer: free once
//               Q K_hat^T of the tile completes) and V_hat^T [128 channels x 128
//               keys] (fp16, double buffer), 128-byte-swizzled K-major, plus the
//               Jensen weights W [4 groups, hi/lo] of the tile; a current-chunk
//               tile is read from global memory (keys converted to fp16, values
//               transposed).
//   warp 12     TMEM owner; lane 0 issues S = Q K_hat^T (fp16, Q converted from
//               bf16 and read from tensor memory), the Jensen term Delta = (q^2) W^T
//               (bf16, N = 16;
//               q^2 of a bf16 q is split exactly into bf16 high and low parts,
//               two MMAs; W columns g and 4 + g hold the high and low bf16 parts
//               of group g's weights), and O += P V_hat with P read from tensor
//               memory (fp16).
// TMEM columns: S double buffer 0-255 (a tile's P overwrites the first 64
// columns of its S once they are read; Q K^T of the tile two later is issued
// only after P V of this one has completed), O 256-383, Delta double buffer
// 384-415 (384-447 in a pair), Q 448-511.  Every wait is bounded; every
// warp-collective tcgen05 load/store runs with the whole warp converged.
//
// CTA pairs (the default): two query tiles of one (batch, head, key-range split)
// run in a 2-CTA cluster whose MMAs have M = 256 (tcgen05 cta_group::2).  Each CTA
// keeps its own 128 rows of Q, S, P, O and the Jensen term, and holds half of
// every B operand: keys 64 r .. 64 r + 63 of the K_hat tile and channels
// 64 r .. 64 r + 63 of the V_hat^T tile (r = the CTA's rank), so each CTA expands
// half of every packed tile -- the expansion per query row is halved.  The even
// CTA issues the MMAs and commits to both CTAs' barriers; the odd CTA's MMA warp
// forwards its K_FULL, V_FULL and P_FULL phases to the even CTA.
//
// Codebook caches ("QuantWM", Methodology: per-channel 4-centroid INT2 keys plus
// the rank-r compensation q . U coeff in the logit): K_hat comes from a byte-permute
// lookup of each key's 2-bit indices in fp16 centroid tables, and the compensation
// is two more fp16 MMAs into S per 16 ranks -- A = U^T q of the query rows (fp32,
// split into fp16 high + low parts, TMEM columns 384-415, where the Jensen term
// lives for INT caches), B = the tile's stored fp16 coefficients.  Codebook keys
// carry no step sizes, so there is no Jensen term for them.
//
// Dequantisation is exact: a code c at bits [b i, b i + b) of a word becomes the
// float c 2^(b i) by or-ing it into the mantissa of 2^23 and subtracting 2^23,
// and fmaf(c 2^(b i), s 2^(-b i), z) rounds c s + z once, as fmaf(c, s, z) does.
// The operands of both products are fp16: K_hat and V_hat are the fp16 roundings
// of the dequantised fp32 entries, Q and the current keys the fp16 conversions of
// their bf16 values (exact inside the fp16 range), P the fp16 rounding of the
// softmax weights.  fp16 keeps 11 significant bits where bf16 keeps 8, which holds
// the logits of keys with large outlier channels within the 16-bit tolerance of the
// exact result.  An entry whose fp16 rounding would be infinite (|x| >= 65520) sets
// the range flag, status word 1.
#include <cstdio>
#include <cstdlib>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace bitkv {

kv_status launch_lse_merge(kv_dtype dt, const float* ws_o, const float2* ws_ml, int n_splits, long long rows, int d,
                           void* out, int out_f32, float* lse, cudaStream_t st);

namespace {

using namespace tc;

constexpr int kM = 128;
constexpr int kN = 128;
constexpr int kD = 128;
constexpr int kSoftWarps = 4;
constexpr int kProdWarps = 8;
constexpr int kProd = 32 * kProdWarps;
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColD = 384, kColQ = 448;
// Single CTA (M = 128) or CTA pair (cta_group::2, M = 256: each CTA's 128 query rows,
// half of every B operand in each CTA: keys 64 r .. 64 r + 63 of K_hat, channels
// 64 r .. 64 r + 63 of V_hat^T, r = the CTA's rank).  The pair's Jensen MMA has N = 32:
// the even CTA holds the 16 weight rows (as a single CTA does), the odd CTA 16 zero rows,
// and the term's TMEM stages are 32 columns apart (384-447, below Q at 448).
template <bool PAIR> struct Geo {
    static constexpr int kKBuf = PAIR ? 2 : 1;       // K_hat (and PSAC coefficient) buffers
    static constexpr int kMM = PAIR ? 256 : 128;     // MMA M
    static constexpr int kNK = PAIR ? 64 : 128;      // K_hat rows (keys) held by this CTA
    static constexpr int kNV = PAIR ? 64 : 128;      // V_hat^T rows (channels) held by this CTA
    static constexpr int kWR = 16;                   // Jensen weight rows held by this CTA
    static constexpr int kJN = PAIR ? 32 : 16;       // Jensen MMA N; TMEM columns per stage
    static constexpr uint32_t kIdescQK = idesc_f16(kMM, kN);   // S = Q K_hat^T (fp16 operands)
    static constexpr uint32_t kIdescJ = idesc_bf16(kMM, kJN);  // Delta = (q^2) W^T
    static constexpr uint32_t kIdescPV = idesc_f16(kMM, kD);   // O += P V_hat (and the PSAC term)
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Cache block formats the kernel reads (one template instance each): INT2 / INT4 with
// fp32 (s, z) pairs, the same with fp16 pairs (H), and codebook blocks.
enum { FMT_INT2 = 0, FMT_INT4 = 1, FMT_CB2 = 2, FMT_INT2H = 3, FMT_INT4H = 4 };
template <int FMT> constexpr int vbits() { return (FMT == FMT_INT4 || FMT == FMT_INT4H) ? 4 : 2; }
template <int FMT> constexpr bool meta_h() { return FMT == FMT_INT2H || FMT == FMT_INT4H; }
template <int FMT> constexpr int pair_bytes() { return meta_h<FMT>() ? 4 : 8; }   // one (s, z)
// bytes of one block (CB2: the largest, PSAC rank 32; the actual stride is the layout's)
template <int FMT> constexpr int max_block_bytes() {
    return FMT == FMT_CB2 ? 24 * kD + kBlockTokens * 32 * 2 : 8 * kD * vbits<FMT>() + 2 * pair_bytes<FMT>() * kD;
}
// byte offsets of the key (step, zero) pairs, the value codes and the value pairs inside a block
template <int FMT> constexpr int koff_meta() { return 4 * kD * vbits<FMT>(); }
template <int FMT> constexpr int voff_codes() {
    return FMT == FMT_CB2 ? 8 * kD : koff_meta<FMT>() + pair_bytes<FMT>() * kD;
}
template <int FMT> constexpr int voff_meta() {
    return FMT == FMT_CB2 ? 16 * kD : voff_codes<FMT>() + 4 * kD * vbits<FMT>();
}
template <int FMT> constexpr int seg_of() { return vbits<FMT>() == 4 ? KV_SEG_INT4 : KV_SEG_INT2; }
constexpr int kCbCoeffOff = 24 * kD;        // CB2: fp16 PSAC coefficients [32][rp]

constexpr int kTile = kM * kD * 2;          // 32 KB: one 16-bit 128 x 128 operand tile
constexpr int kWBytes = 16 * kD * 2;        // 4 KB: 16 x 128 bf16 Jensen weights
constexpr int kExactW = 4 * kD * 4;         // 2 KB: fp32 steps [4 blocks][128] (EXACT Jensen)
constexpr int kCoefTile = kN * 128;         // 16 KB: 128 keys x 64 fp16 PSAC coefficients (swizzled)
constexpr int kCentBytes = kD * 8;          // 1 KB: byte-planar bf16 centroid tables
constexpr int kNumBars = 25;

struct TileInfo {
    int nvalid[4];
    int quantised;
    int pad[3];
    float ss2[4][2];   // ISOTROPIC: sum of s_c^2 of block g over channels 0-63 and 64-127
};

// Shared memory map (bytes from a 1024-aligned base).  INT formats: the bf16 high
// and low parts of q^2 for the Jensen MMA; CB2: the PSAC coefficient tile and the
// centroid tables instead.  In a CTA pair the K_hat, V_hat^T and coefficient tiles
// hold this CTA's half.
template <int FMT, bool PAIR> struct Smem {
    static constexpr bool cb = FMT == FMT_CB2;
    static constexpr int kTileK = Geo<PAIR>::kNK * kD * 2;     // K_hat
    static constexpr int kTileV = Geo<PAIR>::kNV * kN * 2;     // one V_hat^T stage
    static constexpr int q2h = 0;                               // bf16 high part of q^2
    static constexpr int q2l = q2h + (cb ? 0 : kTile);          // low part (q^2 = high + low exactly)
    static constexpr int kTileC = Geo<PAIR>::kNK * 128;        // CB2: PSAC coefficients
    static constexpr int k = q2l + (cb ? 0 : kTile);            // K_hat, kKBuf buffers
    static constexpr int coef = k + Geo<PAIR>::kKBuf * kTileK;  // CB2: PSAC coefficients, kKBuf buffers
    static constexpr int v = coef + (cb ? Geo<PAIR>::kKBuf * kTileC : 0);   // V_hat^T, 2 stages
    static constexpr int w = v + 2 * kTileV;                    // Jensen weights, 2 stages
    static constexpr int cent = w + 2 * kWBytes;                // CB2: centroid tables
    static constexpr int stg = cent + (cb ? kCentBytes : 0);    // staged packed blocks, 2 slots
    static constexpr int stage = 4 * max_block_bytes<FMT>();
    static constexpr int info = stg + 2 * stage;
    static constexpr int stglen = info + 4 * (int)sizeof(TileInfo);   // info: a ring of 4 tiles
    static constexpr int bars = stglen + 2 * 16;
    static constexpr int slot = bars + kNumBars * 8;
    static constexpr int total = slot + 16 + 1024;              // + alignment slack
};

enum {
    BAR_K_FULL = 0,    // [2] producers -> MMA/softmax: K_hat (+ W[s] / PSAC coefficients), info[s] ready
    BAR_V_EMPTY = 2,   // [2] P V of the stage's tile completed
    BAR_S_FULL = 4,    // [2] S and Delta of the tile in TMEM
    BAR_P_FULL = 6,    // [2] softmax -> MMA: P of the stage's tile written
    BAR_O_DONE = 8,    // P V completed
    BAR_K_EMPTY = 9,   // Q K_hat^T completed (K_hat may be overwritten)
    BAR_STG_FULL = 10,   // [2] staging slot filled by the bulk copy
    BAR_STG_EMPTY = 12,  // [2] all producers finished reading the staging slot
    BAR_V_FULL = 14,   // [2] producers -> MMA: V_hat[s] ready
    BAR_MMA_DONE = 16, // every MMA the issuer started has completed (O final; TMEM may be freed)
    BAR_NEVER = 17,    // never arrived on: the target of the injected stall (failure tests)
    // CTA pair, in the even CTA: the odd CTA's K_FULL / V_FULL / P_FULL, forwarded by its
    // MMA warp (the MMAs are issued from the even CTA and read both CTAs' halves)
    BAR_PK_FULL = 18,  // [2]
    BAR_PV_FULL = 20,  // [2]
    BAR_PP_FULL = 22,  // [2]
    BAR_K_EMPTY2 = 24, // CTA pair: Q K_hat^T of a tile in the second K_hat buffer completed
};

// Byte offset of 16-byte chunk `ch` of row `row` in a `rows`-row x 128-column
// 16-bit tile stored as two 64-column, 128-byte-swizzled K-major halves.
__device__ __forceinline__ uint32_t sw_off(int row, int ch, int rows = kM) {
    return (uint32_t)((ch >> 3) * (rows * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// A pair of bf16 values (lower element in the low half) as an fp16 pair, rounded
// to nearest even: exact for magnitudes in [2^-14, 65504] (bf16 carries 8
// significant bits, fp16 11), within 2^-25 below, infinite above.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
    return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// True when either half of an fp16 pair is infinite or NaN.
__device__ __forceinline__ bool h2_nonfinite(uint32_t h) {
    return (h & 0x7C00u) == 0x7C00u || (h & 0x7C000000u) == 0x7C000000u;
}
// The fp16 rounding of x is finite.
__device__ __forceinline__ bool f16_finite(float x) { return fabsf(x) < 65520.0f; }

// 2^e for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// The b-bit code at bits [b i, b i + b) of x as 2^23 + c 2^(b i) (b i + b <= 23): the
// code or-ed into the mantissa of 2^23.
template <int BITS>
__device__ __forceinline__ float code_magic(uint32_t x, int i) {
    return __uint_as_float(0x4B000000u | (x & (((1u << BITS) - 1u) << (BITS * i))));
}

// Two dequantised entries fmaf(c 2^(b i), s 2^(-b i), z) from their magic floats:
// the subtraction of 2^23 is exact, the FMA rounds once.
__device__ __forceinline__ void dequant2(float& v0, float& v1, float m0, float m1, float s0, float s1, float z0,
                                         float z1) {
    float f0, f1;
    add2(f0, f1, m0, m1, -8388608.0f, -8388608.0f);
    fma2(v0, v1, f0, f1, s0, s1, z0, z1);
}

// ------------------------------------------------------------- producers ----
// Values of a staged cache tile into this CTA's V_hat^T rows (fp16; rows = channels,
// K-major along the 128 keys).  Single CTA: warp pw expands value group g = pw & 3
// (channels 32 g .. 32 g + 31, one per lane) of blocks 2 (pw >> 2) and 2 (pw >> 2) + 1.
// CTA pair of rank r: channels 64 r .. 64 r + 63, warp pw takes group 2 r + (pw & 1) of
// block pw >> 1.  fp32 pairs: the group's per-token steps are first pre-scaled in the
// staging copy by 2^(-b i), i = the token's slot in its half word, and each entry is one
// fp32 FMA rounded to fp16.  fp16 pairs: each token pair is one fp16x2 FMA of the exact
// fp16 codes with the tokens' (s, s) and (z, z) pairs -- the entries themselves.
template <int FMT, bool PAIR>
__device__ __forceinline__ void fill_cache_values(unsigned char* Vt, unsigned char* stg, int stride, int nb, int pw,
                                                  int lane, int rank) {
    constexpr int BITS = vbits<FMT>();
    constexpr int kRows = Geo<PAIR>::kNV;
    const int g = PAIR ? 2 * rank + (pw & 1) : (pw & 3), c = 32 * g + lane;
    const int row = (PAIR ? 32 * (pw & 1) : 32 * g) + lane;          // this CTA's tile row
    const int qb = PAIR ? (pw >> 1) : 2 * (pw >> 2);
    constexpr int kNq = PAIR ? 1 : 2;
    constexpr int kSlots = 16 / BITS;    // tokens per half word
#pragma unroll 1
    for (int k2 = 0; k2 < kNq; ++k2) {
        const int q = qb + k2;
        if (q < nb) {
            unsigned char* blk = stg + q * stride;
            const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + voff_codes<FMT>()) + c * BITS;
            if constexpr (meta_h<FMT>()) {
                uint32_t w[BITS];
#pragma unroll
                for (int k = 0; k < BITS; ++k) w[k] = vc[k];
                const uint32_t* vm = reinterpret_cast<const uint32_t*>(blk + voff_meta<FMT>()) + g * 32;
#pragma unroll
                for (int k8 = 0; k8 < 4; ++k8) {     // tokens 8 k8 .. 8 k8 + 7
                    uint32_t h[4];
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const int t = 8 * k8 + i;
                        const uint2 mm = *reinterpret_cast<const uint2*>(vm + t);   // (s, z) of t and t + 1
                        const uint32_t cp = BITS == 2 ? code_pair_f16<2>(w[t >> 4], t & 15)
                                                      : code_pair_f16<4>(w[t >> 3], t & 7);
                        h[i >> 1] = hfma2_u32(cp, __byte_perm(mm.x, mm.y, 0x5410), __byte_perm(mm.x, mm.y, 0x7632));
                    }
                    *reinterpret_cast<uint4*>(Vt + sw_off(row, 4 * q + k8, kRows)) = make_uint4(h[0], h[1], h[2], h[3]);
                }
                continue;
            }
            float* vm = reinterpret_cast<float*>(blk + voff_meta<FMT>()) + g * 64;
            // token t's (s, z) -> (s 2^(-b slot), z), stored per token pair as
            // (s'_t, s'_t+1, z_t, z_t+1) so that pairs load into adjacent registers
            const float2 e = reinterpret_cast<const float2*>(vm)[lane];
            __syncwarp();
            vm[4 * (lane >> 1) + (lane & 1)] = e.x * pow2i(-BITS * (lane % kSlots));
            vm[4 * (lane >> 1) + 2 + (lane & 1)] = e.y;
            __syncwarp();
            uint32_t w[BITS];
#pragma unroll
            for (int k = 0; k < BITS; ++k) w[k] = vc[k];
            const float4* sz = reinterpret_cast<const float4*>(vm);
#pragma unroll
            for (int k8 = 0; k8 < 4; ++k8) {         // tokens 8 k8 .. 8 k8 + 7
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const int t = 8 * k8 + i;
                    const uint32_t x = BITS == 2 ? (w[t >> 4] >> (16 * ((t >> 3) & 1))) : (w[t >> 3] >> (16 * ((t >> 2) & 1)));
                    const float4 p = sz[t >> 1];
                    dequant2(v[i], v[i + 1], code_magic<BITS>(x, t % kSlots), code_magic<BITS>(x, (t + 1) % kSlots),
                             p.x, p.y, p.z, p.w);
                }
                uint4 r;
                r.x = pack_f16(v[0], v[1]);
                r.y = pack_f16(v[2], v[3]);
                r.z = pack_f16(v[4], v[5]);
                r.w = pack_f16(v[6], v[7]);
                *reinterpret_cast<uint4*>(Vt + sw_off(row, 4 * q + k8, kRows)) = r;
            }
        } else {
#pragma unroll
            for (int k8 = 0; k8 < 4; ++k8)
                *reinterpret_cast<uint4*>(Vt + sw_off(row, 4 * q + k8, kRows)) = make_uint4(0, 0, 0, 0);
        }
    }
}

// Key rows of a staged cache tile: thread p expands channels 8 jc .. 8 jc + 7 (jc = p & 15)
// of NR consecutive keys of one block into K_hat (fp16).  Single CTA: 8 keys per thread,
// the tile's 128 keys; CTA pair of rank r: 4 keys per thread, keys 64 r .. 64 r + 63
// (blocks 2 r and 2 r + 1).  *q, *t0, *row0: the block, its first token, the tile row.
template <bool PAIR>
__device__ __forceinline__ void key_rows(int p, int rank, int* q, int* t0, int* row0) {
    if (PAIR) {
        const int kg = (p >> 4) & 7, rh = p >> 7, ql = kg >> 2;
        *q = 2 * rank + ql;
        *t0 = 8 * (kg & 3) + 4 * rh;
        *row0 = 32 * ql + *t0;
    } else {
        const int kg = p >> 4;
        *q = kg >> 2;
        *t0 = 8 * (kg & 3);
        *row0 = 32 * *q + *t0;
    }
}

template <int FMT, bool PAIR>
__device__ __forceinline__ void fill_cache_keys(unsigned char* Kt, const unsigned char* stg, int nb, int p, int rank) {
    constexpr int BITS = vbits<FMT>();
    constexpr int NR = PAIR ? 4 : 8, kRows = Geo<PAIR>::kNK;
    const int jc = p & 15;
    int q, t0, row0;
    key_rows<PAIR>(p, rank, &q, &t0, &row0);
    if (q >= nb) {
#pragma unroll
        for (int r = 0; r < NR; ++r) *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r, jc, kRows)) = make_uint4(0, 0, 0, 0);
        return;
    }
    const unsigned char* blk = stg + q * max_block_bytes<FMT>();
    constexpr int KW = kD * BITS / 32;   // code words per key
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk);
    if constexpr (meta_h<FMT>()) {
        // fp16 pairs: channel pairs' (s, s) and (z, z), then one fp16x2 FMA per entry pair
        const uint4* km = reinterpret_cast<const uint4*>(blk + koff_meta<FMT>()) + 2 * jc;
        const uint4 m0 = km[0], m1 = km[1];
        const uint32_t m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        uint32_t sp[4], zp[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sp[i] = __byte_perm(m[2 * i], m[2 * i + 1], 0x5410);
            zp[i] = __byte_perm(m[2 * i], m[2 * i + 1], 0x7632);
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int t = t0 + r;
            const uint32_t x = BITS == 2 ? kc[t * KW + (jc >> 1)] >> (16 * (jc & 1)) : kc[t * KW + jc];
            uint4 rr;
            rr.x = hfma2_u32(code_pair_f16<BITS>(x, 0), sp[0], zp[0]);
            rr.y = hfma2_u32(code_pair_f16<BITS>(x, 2), sp[1], zp[1]);
            rr.z = hfma2_u32(code_pair_f16<BITS>(x, 4), sp[2], zp[2]);
            rr.w = hfma2_u32(code_pair_f16<BITS>(x, 6), sp[3], zp[3]);
            *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r, jc, kRows)) = rr;
        }
        return;
    }
    constexpr int kSlots = 16 / BITS;
    float s[8], z[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 v = meta2_at<meta_h<FMT>()>(blk + koff_meta<FMT>(), 8 * jc + 2 * k);
        s[2 * k] = v.x;
        z[2 * k] = v.y;
        s[2 * k + 1] = v.z;
        z[2 * k + 1] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] *= pow2i(-BITS * (i % kSlots));
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int t = t0 + r;
        float v[8];
        if (BITS == 2) {
            const uint32_t x = kc[t * KW + (jc >> 1)] >> (16 * (jc & 1));
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                dequant2(v[i], v[i + 1], code_magic<2>(x, i), code_magic<2>(x, i + 1), s[i], s[i + 1], z[i], z[i + 1]);
        } else {
            const uint32_t w = kc[t * KW + jc];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const uint32_t x = i < 4 ? w : (w >> 16);
                dequant2(v[i], v[i + 1], code_magic<4>(x, i & 3), code_magic<4>(x, (i + 1) & 3), s[i], s[i + 1], z[i],
                         z[i + 1]);
            }
        }
        uint4 rr;
        rr.x = pack_f16(v[0], v[1]);
        rr.y = pack_f16(v[2], v[3]);
        rr.z = pack_f16(v[4], v[5]);
        rr.w = pack_f16(v[6], v[7]);
        *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r, jc, kRows)) = rr;
    }
}

// Centroid tables of one (batch, kv head) for the codebook key lookup: channel c's
// four centroids rounded to fp16, stored byte-planar as two words -- the four low
// bytes, then the four high bytes -- so that one byte permute with selector
// nibbles (k, 4 + k) returns centroid k as an fp16.  Returns false if a centroid's
// fp16 rounding is not finite.
__device__ __forceinline__ bool fill_centroid_tables(uint32_t* tab, const float* cent, int tid) {
    bool ok = true;
    for (int ch = tid; ch < kD; ch += kThreads) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(cent) + ch);
        ok = ok && f16_finite(v.x) && f16_finite(v.y) && f16_finite(v.z) && f16_finite(v.w);
        const uint32_t c01 = pack_f16(v.x, v.y), c23 = pack_f16(v.z, v.w);
        tab[2 * ch] = __byte_perm(c01, c23, 0x6420);
        tab[2 * ch + 1] = __byte_perm(c01, c23, 0x7531);
    }
    return ok;
}

// Keys of a staged codebook tile (the rows of fill_cache_keys) into K_hat (fp16) by
// looking the 2-bit centroid indices up in the channels' tables, two keys at a time.
// For the channel pair (2 i, 2 i + 1) the four index bits n = k0 + 4 k1 of a key become
// the selector bytes (17 k0 + 0x40, 17 k1 + 0x40), i.e. nibbles (k0, 4 + k0, k1, 4 + k1):
// 17 n + 1071 (n & 12) + 0x4040 = 17 k0 + 4352 k1 + 0x4040.
template <bool PAIR>
__device__ __forceinline__ void fill_cb_keys(unsigned char* Kt, const unsigned char* stg, int stride, int nb,
                                             const uint32_t* tab, int p, int rank) {
    constexpr int NR = PAIR ? 4 : 8, kRows = Geo<PAIR>::kNK;
    const int jc = p & 15;
    int q, t0, row0;
    key_rows<PAIR>(p, rank, &q, &t0, &row0);
    if (q >= nb) {
#pragma unroll
        for (int r = 0; r < NR; ++r) *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r, jc, kRows)) = make_uint4(0, 0, 0, 0);
        return;
    }
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 v = reinterpret_cast<const uint4*>(tab)[4 * jc + k];
        lo[2 * k] = v.x;
        hi[2 * k] = v.y;
        lo[2 * k + 1] = v.z;
        hi[2 * k + 1] = v.w;
    }
    constexpr int KW = kD / 16;   // code words per key
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(stg + q * stride);
    const uint32_t half = (jc & 1) ? 0x7632u : 0x5410u;
#pragma unroll
    for (int r = 0; r < NR; r += 2) {
        const int t = t0 + r;
        // key t's 8 indices in the low half, key t + 1's in the high half
        const uint32_t x = __byte_perm(kc[t * KW + (jc >> 1)], kc[(t + 1) * KW + (jc >> 1)], half);
        uint32_t o0[4], o1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t y = x >> (4 * i);
            const uint32_t sel = (y & 0x000F000Fu) * 17u + (y & 0x000C000Cu) * 1071u + 0x40404040u;
            const uint32_t sel1 = sel >> 16;
            o0[i] = __byte_perm(__byte_perm(lo[2 * i], hi[2 * i], sel), __byte_perm(lo[2 * i + 1], hi[2 * i + 1], sel),
                                0x7610);
            o1[i] = __byte_perm(__byte_perm(lo[2 * i], hi[2 * i], sel1),
                                __byte_perm(lo[2 * i + 1], hi[2 * i + 1], sel1), 0x7610);
        }
        *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r, jc, kRows)) = make_uint4(o0[0], o0[1], o0[2], o0[3]);
        *reinterpret_cast<uint4*>(Kt + sw_off(row0 + r + 1, jc, kRows)) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    }
}

// PSAC coefficients of a staged codebook tile -> the K-major swizzled B operand
// [this CTA's keys x nch 8-element chunks] (fp16); chunks at or beyond the stored rp
// and rows of missing blocks are zero.
template <bool PAIR>
__device__ __forceinline__ void fill_coeff(unsigned char* Ct, const unsigned char* stg, int stride, int nb, int rp,
                                           int nch, int p, int rank) {
    constexpr int kRows = Geo<PAIR>::kNK;
    const int qbase = PAIR ? 2 * rank : 0;
    for (int e = p; e < kRows * nch; e += kProd) {
        const int row = e / nch, ch = e - (e / nch) * nch, q = qbase + (row >> 5), t = row & 31;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (q < nb && 8 * ch < rp)
            v = *reinterpret_cast<const uint4*>(stg + q * stride + kCbCoeffOff + (t * rp + 8 * ch) * 2);
        *reinterpret_cast<uint4*>(Ct + sw_off(row, ch, kRows)) = v;
    }
}

// Jensen weights of a staged tile.  TAYLOR2: W rows g and 4 + g hold the bf16 high and
// low parts of w_c = s_c^2 tau^2 / 24 log2(e) of block g (zero for missing blocks); the
// other rows stay zero (`wrows` rows in the tile).  EXACT: the block steps s_c as fp32 [4][128].
// ISOTROPIC: the two warps of block g each sum s_c^2 over their 64 channels into
// ss2[g][w] (the softmax adds the two in a fixed order).
template <int FMT, int JENSEN>
__device__ __forceinline__ void fill_weights(unsigned char* W, const unsigned char* stg, int nb, int p, float coef,
                                             int wrows, float (*ss2)[2] = nullptr) {
    const int g = p >> 6, c = 2 * (p & 63);
    float2 s = make_float2(0.0f, 0.0f);
    if (g < nb) {
        const float4 v = meta2_at<meta_h<FMT>()>(stg + g * max_block_bytes<FMT>() + koff_meta<FMT>(), c);
        s = make_float2(v.x, v.z);
    }
    if (JENSEN == KV_JENSEN_TAYLOR2) {
        const float w0 = s.x * s.x * coef, w1 = s.y * s.y * coef;
        const uint32_t hi = pack_bf16(w0, w1);
        const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
        const uint32_t lo = pack_bf16(w0 - h0, w1 - h1);
        const int cb = (c & 7) * 2;
        *reinterpret_cast<uint32_t*>(W + sw_off(g, c >> 3, wrows) + cb) = hi;
        *reinterpret_cast<uint32_t*>(W + sw_off(4 + g, c >> 3, wrows) + cb) = lo;
    } else if (JENSEN == KV_JENSEN_EXACT) {
        reinterpret_cast<float2*>(W)[(g * kD + c) >> 1] = s;
    } else if (JENSEN == KV_JENSEN_ISOTROPIC) {
        const float v = warp_sum(fmaf(s.x, s.x, s.y * s.y));
        if ((p & 31) == 0) ss2[g][(p >> 5) & 1] = v;
    }
}

// Current-chunk tile (unquantised bf16): values transposed to fp16 V_hat^T rows.  Each
// thread transposes one 8 x 8 block (keys 8 kc8 .., channels 8 cch ..): single CTA all
// 128 channels (16 chunks); pair of rank r its 64 (8 chunks, threads 0-127).
template <bool PAIR>
__device__ __forceinline__ void fill_current_values(unsigned char* Vt, const __nv_bfloat16* Vcur, long long row0,
                                                    int valid, int p, int rank) {
    constexpr int kRows = Geo<PAIR>::kNV;
    if (PAIR && p >= 128) return;
    const uint4* Vg = reinterpret_cast<const uint4*>(Vcur + row0 * kD);
    const int kc8 = PAIR ? (p >> 3) : (p >> 4), cch = PAIR ? (p & 7) : (p & 15);
    const int gch = PAIR ? 8 * rank + cch : cch;     // the 16-byte chunk of the key row
    uint32_t x[8][4];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int key = 8 * kc8 + k;
        const uint4 v = key < valid ? __ldg(Vg + key * (kD / 8) + gch) : make_uint4(0, 0, 0, 0);
        x[k][0] = v.x;
        x[k][1] = v.y;
        x[k][2] = v.z;
        x[k][3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // channel 8 gch + i: element i of every key row (word i / 2, half i & 1)
        const int wi = i >> 1, hf = i & 1;
        float f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(hf ? (x[k][wi] & 0xFFFF0000u) : (x[k][wi] << 16));
        uint4 y;
        y.x = pack_f16(f[0], f[1]);
        y.y = pack_f16(f[2], f[3]);
        y.z = pack_f16(f[4], f[5]);
        y.w = pack_f16(f[6], f[7]);
        *reinterpret_cast<uint4*>(Vt + sw_off(8 * cch + i, kc8, kRows)) = y;
    }
}

// Current-chunk keys: bf16 rows converted to fp16 into the swizzled K_hat buffer (pair of
// rank r: keys 64 r .. 64 r + 63).  Returns false if a key's fp16 rounding is not finite.
template <bool PAIR>
__device__ __forceinline__ bool fill_current_keys(unsigned char* Kt, const __nv_bfloat16* Kcur, long long row0,
                                                  int valid, int p, int rank) {
    constexpr int kRows = Geo<PAIR>::kNK, NI = kRows / 16;
    const int jc = p & 15, r0 = p >> 4, kb = PAIR ? 64 * rank : 0;
    const uint4* Kg = reinterpret_cast<const uint4*>(Kcur + row0 * kD);
    uint4 kv[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int key = kb + r0 + 16 * i;
        kv[i] = key < valid ? __ldg(Kg + key * (kD / 8) + jc) : make_uint4(0, 0, 0, 0);
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const uint4 h = make_uint4(bf2_to_h2(kv[i].x), bf2_to_h2(kv[i].y), bf2_to_h2(kv[i].z), bf2_to_h2(kv[i].w));
        bad |= h2_nonfinite(h.x) | h2_nonfinite(h.y) | h2_nonfinite(h.z) | h2_nonfinite(h.w);
        *reinterpret_cast<uint4*>(Kt + sw_off(r0 + 16 * i, jc, kRows)) = h;
    }
    return !bad;
}

// The cached keys of a staged INT tile stay inside the fp16 range: every entry of a
// (block, channel) lies between z and fmaf(2^b - 1, s, z), so checking those two
// bounds for each of the thread's two channels covers the tile.
template <int FMT>
__device__ __forceinline__ bool cache_keys_in_f16_range(const unsigned char* stg, int nb, int p) {
    const int g = p >> 6, c = 2 * (p & 63);
    if (g >= nb) return true;
    const float4 v = meta2_at<meta_h<FMT>()>(stg + g * max_block_bytes<FMT>() + koff_meta<FMT>(), c);
    constexpr float kTop = (float)((1 << vbits<FMT>()) - 1);
    return f16_finite(v.y) && f16_finite(fmaf(kTop, v.x, v.y)) && f16_finite(v.w) && f16_finite(fmaf(kTop, v.z, v.w));
}

// --------------------------------------------------------------- kernel -----
template <int FMT, int JENSEN, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kcur,
               const __nv_bfloat16* __restrict__ Vcur, int n_q, int n_cur, int Hq, DevCache c, float tau, int r16,
               int n_splits, void* __restrict__ out, int out_f32, float* __restrict__ lse, float* __restrict__ ws_o,
               float2* __restrict__ ws_ml, int* __restrict__ err, int stall) {
    using M = Smem<FMT, PAIR>;
    using G = Geo<PAIR>;
    constexpr bool kCb = FMT == FMT_CB2;
    extern __shared__ unsigned char smem_raw[];
    __shared__ volatile int abort_flag;
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_qt = (n_q + kM - 1) / kM;
    // a CTA pair takes two query tiles of one (batch, head, split); with an odd tile count
    // the last pair's odd CTA has no valid row and only contributes its operand halves
    const int rank = PAIR ? (int)cluster_rank() : 0;
    const int n_qp = (n_qt + 1) / 2;
    const int qt = PAIR ? 2 * ((blockIdx.x >> 1) % n_qp) + rank : blockIdx.x % n_qt;
    const int split = PAIR ? (int)(blockIdx.x >> 1) / n_qp : blockIdx.x / n_qt;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int h = hq / (Hq / c.Hkv);
    const int q0 = qt * kM;
    const int seg = seg_of<FMT>();
    // staging stride of one block (a CB2 block's size depends on the PSAC rank)
    const int bb = kCb ? (int)c.block_bytes[seg] : max_block_bytes<FMT>();
    const int n_cache_tiles = (c.n_blocks[seg] + 3) / 4;
    const int n_tiles = n_cache_tiles + (n_cur + kN - 1) / kN;
    // split s takes tiles s, s + n_splits, ...: every split gets an even share of
    // cache and current-chunk tiles, and its cache tiles still come first.
    const int T = split < n_tiles ? (n_tiles - split + n_splits - 1) / n_splits : 0;
    auto tile_of = [&](int j) { return split + j * n_splits; };
    auto bar = [&](int i) { return sbase + M::bars + 8 * i; };
    TileInfo* infos = reinterpret_cast<TileInfo*>(sm + M::info);
    const int nblk = c.n_blocks[seg];
    int* stg_len = reinterpret_cast<int*>(sm + M::stglen);
    // Bulk-copy cache tile j (if it is one) into staging slot j & 1, with its
    // blocks' valid lengths: tiles 0 and 1 by thread 0 after the barriers are
    // initialised, later ones by producer thread 0 two tiles ahead.
    auto stage_copy = [&](int j) {
        const int tile = tile_of(j);
        if (j >= T || tile >= n_cache_tiles) return;
        const int nb = min(4, nblk - tile * 4);
        for (int q = 0; q < 4; ++q)
            stg_len[(j & 1) * 4 + q] = q < nb ? c.blk_len[(long long)b * c.cap_total + c.seg_base[seg] + tile * 4 + q] : 0;
        const uint32_t bytes = (uint32_t)(nb * bb);
        const uint32_t sbar = bar(BAR_STG_FULL + (j & 1));
        mbar_expect_tx(sbar, bytes);
        bulk_g2s(sbase + M::stg + (j & 1) * M::stage, block_ptr(c, b, h, seg, tile * 4), bytes, sbar);
    };

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar(BAR_K_FULL + 0), kProd);
        mbar_init(bar(BAR_K_FULL + 1), kProd);
        mbar_init(bar(BAR_V_FULL + 0), kProd);
        mbar_init(bar(BAR_V_FULL + 1), kProd);
        mbar_init(bar(BAR_MMA_DONE), 1);
        mbar_init(bar(BAR_NEVER), 1);
        mbar_init(bar(BAR_V_EMPTY + 0), 1);
        mbar_init(bar(BAR_V_EMPTY + 1), 1);
        mbar_init(bar(BAR_S_FULL + 0), 1);
        mbar_init(bar(BAR_S_FULL + 1), 1);
        mbar_init(bar(BAR_P_FULL + 0), 32 * kSoftWarps);
        mbar_init(bar(BAR_P_FULL + 1), 32 * kSoftWarps);
        mbar_init(bar(BAR_O_DONE), 1);
        mbar_init(bar(BAR_K_EMPTY), 1);
        mbar_init(bar(BAR_STG_FULL + 0), 1);
        mbar_init(bar(BAR_STG_FULL + 1), 1);
        mbar_init(bar(BAR_STG_EMPTY + 0), kProd);
        mbar_init(bar(BAR_STG_EMPTY + 1), kProd);
        for (int i = 0; i < 7; ++i) mbar_init(bar(BAR_PK_FULL + i), 1);   // PK, PV, PP, K_EMPTY2
        mbar_fence_init();
        // the first two cache tiles' copies start now, under the prologue
        stage_copy(0);
        stage_copy(1);
    }
    if (warp == kMmaWarp) {
        if (PAIR) tmem_alloc2(sbase + M::slot, kTmemCols);
        else tmem_alloc(sbase + M::slot, kTmemCols);
    }

    const uint4* Qg = reinterpret_cast<const uint4*>(Q + (((long long)b * Hq + hq) * n_q) * kD);
    // PSAC basis U of this head, zero-padded to [d][r16] fp32, staged in the second
    // V_hat stage (written by the producers only after the second barrier below)
    float* Us = reinterpret_cast<float*>(sm + M::v + M::kTileV);
    if (kCb) {
        if (!fill_centroid_tables(reinterpret_cast<uint32_t*>(sm + M::cent),
                                  c.centroids + ((long long)b * c.Hkv + h) * kD * 4, tid))
            atomicExch(err + 1, 1);
        if (r16 > 0) {
            const float* U = c.psac_u + ((long long)b * c.Hkv + h) * kD * c.r;
            for (int e = tid; e < kD * r16; e += kThreads) {
                const int ch = e / r16, jj = e - (e / r16) * r16;
                Us[e] = jj < c.r ? __ldg(U + ch * c.r + jj) : 0.0f;
            }
        }
    } else {
        // q^2 of the Q tile (bf16 q, so q^2 has at most 16 significant bits and splits
        // exactly into bf16 high + low) -> swizzled smem, rows beyond n_q zero; the
        // Jensen weight tiles start zero (rows 8-15 stay zero).  EXACT: the bf16 rows of q
        // themselves in the high part's place, read by the softmax for every cache tile.
        for (int e = tid; e < kM * kD / 8; e += kThreads) {
            const int row = e >> 4, ch = e & 15;
            const uint4 v =
                (q0 + row < n_q) ? __ldg(Qg + (long long)(q0 + row) * (kD / 8) + ch) : make_uint4(0, 0, 0, 0);
            if (JENSEN == KV_JENSEN_EXACT) {
                *reinterpret_cast<uint4*>(sm + M::q2h + sw_off(row, ch)) = v;
                continue;
            }
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t hq2[4], lq2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = __uint_as_float(wv[k] << 16), hi = __uint_as_float(wv[k] & 0xFFFF0000u);
                const float a = lo * lo, bq = hi * hi;
                hq2[k] = pack_bf16(a, bq);
                lq2[k] = pack_bf16(a - __uint_as_float(hq2[k] << 16), bq - __uint_as_float(hq2[k] & 0xFFFF0000u));
            }
            *reinterpret_cast<uint4*>(sm + M::q2h + sw_off(row, ch)) = make_uint4(hq2[0], hq2[1], hq2[2], hq2[3]);
            *reinterpret_cast<uint4*>(sm + M::q2l + sw_off(row, ch)) = make_uint4(lq2[0], lq2[1], lq2[2], lq2[3]);
        }
        for (int e = tid; e < 2 * kWBytes / 16; e += kThreads)
            reinterpret_cast<uint4*>(sm + M::w)[e] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async();
    fence_before();
    __syncthreads();
    // a pair's barriers are initialised in both CTAs before either signals the other
    if (PAIR) cluster_sync();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + M::slot);
    // codebook keys with residual variances: the Jensen term of this thread's query row,
    // (tau^2/2) log2(e) sum_c q'_c^2 v_c (ISOTROPIC: |q'|^2 mean_c v_c), q' = q - U (U^T q)
    // with the PSAC term on, the same for every cached key
    float jrow = 0.0f;
    if (warp < kSoftWarps) {
        // Q row i -> TMEM lane i, columns kColQ .. kColQ + 63 (two fp16 per column: the
        // bf16 queries converted, exactly inside the fp16 range)
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const bool valid = q0 + tid < n_q;
        bool qbad = false;
#pragma unroll
        for (int hf = 0; hf < 4; ++hf) {
            uint32_t u[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = valid ? __ldg(Qg + (long long)(q0 + tid) * (kD / 8) + 4 * hf + k) : make_uint4(0, 0, 0, 0);
                u[4 * k] = bf2_to_h2(v.x);
                u[4 * k + 1] = bf2_to_h2(v.y);
                u[4 * k + 2] = bf2_to_h2(v.z);
                u[4 * k + 3] = bf2_to_h2(v.w);
#pragma unroll
                for (int e = 0; e < 4; ++e) qbad |= h2_nonfinite(u[4 * k + e]);
            }
            tmem_st16(tmem + lane_addr + kColQ + 16 * hf, u);
        }
        if (qbad) atomicExch(err + 1, 1);
        float uall[32];
        if (kCb && r16 > 0) {
            // u = U^T q of row i in fp32, split into fp16 high + low parts (u = hi + lo up
            // to 2^-22 |u|): the A operand of the PSAC MMAs, TMEM columns kColD + 8 ks
            // (high) and kColD + 16 + 8 ks (low) for the 16-wide rank chunk ks
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                if (ks >= r16 / 16) break;
                float u[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) u[jj] = 0.0f;
#pragma unroll 1
                for (int c8 = 0; c8 < kD / 8; ++c8) {
                    const uint4 v = valid ? __ldg(Qg + (long long)(q0 + tid) * (kD / 8) + c8) : make_uint4(0, 0, 0, 0);
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float qf = __uint_as_float(k & 1 ? (wv[k >> 1] & 0xFFFF0000u) : (wv[k >> 1] << 16));
                        const float4* ur = reinterpret_cast<const float4*>(Us + (8 * c8 + k) * r16 + 16 * ks);
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const float4 w4 = ur[j4];
                            u[4 * j4] = fmaf(w4.x, qf, u[4 * j4]);
                            u[4 * j4 + 1] = fmaf(w4.y, qf, u[4 * j4 + 1]);
                            u[4 * j4 + 2] = fmaf(w4.z, qf, u[4 * j4 + 2]);
                            u[4 * j4 + 3] = fmaf(w4.w, qf, u[4 * j4 + 3]);
                        }
                    }
                }
                if (JENSEN != KV_JENSEN_OFF) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) uall[16 * ks + jj] = u[jj];
                }
                uint32_t uh[8], ul[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uh[k] = pack_f16(u[2 * k], u[2 * k + 1]);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&uh[k]));
                    ul[k] = pack_f16(u[2 * k] - hf.x, u[2 * k + 1] - hf.y);
                }
                tmem_st8(tmem + lane_addr + kColD + 8 * ks, uh);
                tmem_st8(tmem + lane_addr + kColD + 16 + 8 * ks, ul);
            }
        }
        if (kCb && JENSEN != KV_JENSEN_OFF) {
            const float* vv = c.resid_var + ((long long)b * c.Hkv + h) * kD;
            float acc = 0.0f, qn = 0.0f, vs = 0.0f;
#pragma unroll 1
            for (int c8 = 0; c8 < kD / 8; ++c8) {
                const uint4 v = valid ? __ldg(Qg + (long long)(q0 + tid) * (kD / 8) + c8) : make_uint4(0, 0, 0, 0);
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int ch = 8 * c8 + k;
                    float qc = __uint_as_float(k & 1 ? (wv[k >> 1] & 0xFFFF0000u) : (wv[k >> 1] << 16));
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (jj < r16) qc = fmaf(-Us[ch * r16 + jj], uall[jj], qc);
                    const float var = __ldg(vv + ch);
                    acc = fmaf(qc * qc, var, acc);
                    qn = fmaf(qc, qc, qn);
                    vs += var;
                }
            }
            const float jc = 0.5f * tau * tau * kLog2e;
            jrow = JENSEN == KV_JENSEN_ISOTROPIC ? jc * qn * (vs * (1.0f / kD)) : jc * acc;
        }
        tmem_wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();

    if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && rank == 0) {
            const uint32_t sQ2h = sbase + M::q2h, sQ2l = sbase + M::q2l, sK = sbase + M::k;
            auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t bd, uint32_t id, uint32_t acc) {
                if (PAIR) mma_f16kind_ts2(d, a, bd, id, acc);
                else mma_f16kind_ts(d, a, bd, id, acc);
            };
            auto commit = [&](uint32_t bq) {
                if (PAIR) mma_commit2(bq);
                else mma_commit(bq);
            };
            auto issue_qk = [&](int j) {
                const int s = j & 1;
                const uint32_t sKb = sK + (PAIR ? s * M::kTileK : 0);
                fence_after();
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (G::kNK * 128) + (kk & 3) * 32;
                    mma_ts(tmem + kColS + s * kN, tmem + kColQ + 8 * kk, desc_sw128(sKb + off), G::kIdescQK, kk > 0);
                }
                if (kCb && r16 > 0 && tile_of(j) < n_cache_tiles) {
                    // S += (U^T q) coeff^T: fp16, K = the rank padded to 16, high and low
                    // parts of U^T q against the same coefficients
                    const uint32_t sC = sbase + M::coef + (PAIR ? s * M::kTileC : 0);
                    for (int ks = 0; ks < r16 / 16; ++ks) {
                        mma_ts(tmem + kColS + s * kN, tmem + kColD + 8 * ks, desc_sw128(sC + 32 * ks), G::kIdescPV, 1);
                        mma_ts(tmem + kColS + s * kN, tmem + kColD + 16 + 8 * ks, desc_sw128(sC + 32 * ks), G::kIdescPV,
                               1);
                    }
                }
                if (!kCb && JENSEN == KV_JENSEN_TAYLOR2 && tile_of(j) < n_cache_tiles) {
                    const uint32_t sW = sbase + M::w + s * kWBytes;
#pragma unroll
                    for (int kk = 0; kk < 2 * (kD / 16); ++kk) {
                        const int k = kk & 7;
                        const uint32_t offa = (k >> 2) * (kM * 128) + (k & 3) * 32;
                        const uint32_t offb = (k >> 2) * (G::kWR * 128) + (k & 3) * 32;
                        const uint64_t ad = desc_sw128((kk < 8 ? sQ2h : sQ2l) + offa), bd = desc_sw128(sW + offb);
                        if (PAIR) mma_f16kind2(tmem + kColD + G::kJN * s, ad, bd, G::kIdescJ, kk > 0);
                        else mma_f16kind(tmem + kColD + G::kJN * s, ad, bd, G::kIdescJ, kk > 0);
                    }
                }
                commit(bar(BAR_S_FULL + s));
                commit(bar(PAIR && s ? BAR_K_EMPTY2 : BAR_K_EMPTY));
            };
            auto issue_pv = [&](int jj) {
                fence_after();
                const uint32_t sV = sbase + M::v + (jj & 1) * M::kTileV;
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (G::kNV * 128) + (kk & 3) * 32;
                    mma_ts(tmem + kColO, tmem + kColS + (jj & 1) * kN + 8 * kk, desc_sw128(sV + off), G::kIdescPV,
                           (jj > 0 || kk > 0));
                }
                commit(bar(BAR_O_DONE));
                commit(bar(BAR_V_EMPTY + (jj & 1)));
            };
            // the odd CTA's halves, forwarded by its MMA warp (a pair only): polled relaxed,
            // one acquire fence before the MMAs that read them are issued
            auto peer = [&](int base, int j) {
                return !PAIR || mbar_test_wait_relaxed_cluster(bar(base + (j & 1)), (j >> 1) & 1);
            };
            // Issue Q K^T of tile j as soon as its operands are staged and P V of
            // tile i as soon as its P is written, whichever is ready first (P V of a
            // tile frees the V stage the producers refill next).  Q K^T of tile j
            // writes the S columns that P V of tile j - 2 reads its P from.  MMAs into
            // different accumulators are not ordered with one another, so Q K^T of
            // tile j waits until P V of tile j - 2 has completed (its V stage's empty
            // barrier, which nothing else can have advanced past it yet); that wait also
            // keeps Q K^T at most one tile ahead of the P V issued so far.  The wait is
            // bounded: no progress for ~2^30 cycles gives up.
            int nq = 0, np = 0;
            long long t_prog = clock64();
            while (np < T) {
                bool progressed = false;
                if (np < nq && mbar_test_wait(bar(BAR_P_FULL + (np & 1)), (np >> 1) & 1) &&
                    mbar_test_wait(bar(BAR_V_FULL + (np & 1)), (np >> 1) & 1) && peer(BAR_PP_FULL, np) &&
                    peer(BAR_PV_FULL, np)) {
                    if (PAIR) fence_acquire_cluster();
                    issue_pv(np++);
                    progressed = true;
                } else if (nq < T && nq <= np + 1 && mbar_test_wait(bar(BAR_K_FULL + (nq & 1)), (nq >> 1) & 1) &&
                           peer(BAR_PK_FULL, nq) &&
                           (nq < 2 || mbar_test_wait(bar(BAR_V_EMPTY + (nq & 1)), ((nq - 2) >> 1) & 1))) {
                    if (PAIR) fence_acquire_cluster();
                    issue_qk(nq++);
                    progressed = true;
                }
                if (progressed) {
                    t_prog = clock64();
                } else if (abort_flag) {
                    break;
                } else if (clock64() - t_prog > 1000000000LL) {
                    abort_flag = 1;
                    atomicExch(err, 1);
                    break;
                }
            }
            // every MMA issued so far completes before TMEM is freed (also after an abort)
            commit(bar(BAR_MMA_DONE));
            const long long t_done = clock64();
            while (!mbar_try_wait(bar(BAR_MMA_DONE), 0) && clock64() - t_done < 100000000LL) {
            }
        } else if (PAIR && rank == 1 && lane < 3) {
            // the odd CTA of a pair: lanes 0, 1 and 2 forward this CTA's K_FULL, V_FULL and
            // P_FULL phases to the even CTA, whose MMAs read this CTA's halves; one lane per
            // barrier, so that a forward waits for no other.  No phase can run two ahead of its forwarding: K_FULL of tile
            // j + 2 needs this CTA's P_FULL of tile j, V_FULL of j + 2 the completion of
            // P V of j, P_FULL of j + 2 the Q K^T of j + 2, each issued only after tile j's
            // phase was forwarded.
            const int lb = lane == 0 ? BAR_K_FULL : (lane == 1 ? BAR_V_FULL : BAR_P_FULL);
            const int rb = lane == 0 ? BAR_PK_FULL : (lane == 1 ? BAR_PV_FULL : BAR_PP_FULL);
            int f = 0;
            long long t_prog = clock64();
            while (f < T) {
                if (mbar_test_wait(bar(lb + (f & 1)), (f >> 1) & 1)) {
                    mbar_arrive_remote(bar(rb + (f & 1)), 0);
                    ++f;
                    t_prog = clock64();
                } else if (abort_flag) {
                    break;
                } else if (clock64() - t_prog > 1000000000LL) {
                    abort_flag = 1;
                    atomicExch(err, 3);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= kSoftWarps) {
        // ----------------------------------------------------------- producers
        const int p = tid - 32 * kSoftWarps, pw = p >> 5;
        const float jcoef = tau * tau * (1.0f / 24.0f) * kLog2e;
        int issued = min(T, 2);   // staging copies issued so far (tiles 0 and 1 by thread 0)
        int j = 0;
        for (; j < T; ++j) {
            const int s = j & 1;
            const int tile = tile_of(j);
            const bool cached = tile < n_cache_tiles;
            // keys first: a single K_hat buffer (and W[s], the PSAC coefficients) is free
            // once Q K_hat^T of tile j - 1 completed; with two (a CTA pair), buffer j & 1
            // once Q K_hat^T of tile j - 2 completed, signalled on that buffer's own barrier
            // (one barrier for both could not express tile j - 2 once j - 1 completed too)
            bool ok = true;
            if (cached) ok = mbar_wait(bar(BAR_STG_FULL + s), (j >> 1) & 1, &abort_flag, err, 9);
            if (PAIR) {
                if (ok && j >= 2)
                    ok = mbar_wait(bar(s ? BAR_K_EMPTY2 : BAR_K_EMPTY), ((j - 2) >> 1) & 1, &abort_flag, err, 8);
            } else if (ok && j > 0) {
                ok = mbar_wait(bar(BAR_K_EMPTY), (j - 1) & 1, &abort_flag, err, 8);
            }
            unsigned char* Kt = sm + M::k + (PAIR ? s * M::kTileK : 0);
            unsigned char* Ct = sm + M::coef + (PAIR ? s * M::kTileC : 0);
            if (!__all_sync(0xffffffffu, ok)) break;
            unsigned char* stg = sm + M::stg + s * M::stage;
            const int nb = cached ? min(4, nblk - tile * 4) : 0;
            const int t0 = (tile - n_cache_tiles) * kN;
            const long long row0 = ((long long)b * c.Hkv + h) * n_cur + t0;
            const int cvalid = min(kN, n_cur - t0);
            // tile info in a ring of 4: the softmax read tile j - 4's copy before P V of
            // tile j - 3 was issued, which Q K^T of tile j - 1 waited for
            TileInfo& inf = infos[j & 3];
            if (p < 4) inf.nvalid[p] = cached ? (p < nb ? stg_len[s * 4 + p] : 0) : min(32, max(0, cvalid - 32 * p));
            if (p == 0) inf.quantised = cached ? 1 : 0;
            if (cached && kCb) {
                fill_cb_keys<PAIR>(Kt, stg, bb, nb, reinterpret_cast<const uint32_t*>(sm + M::cent), p, rank);
                if (r16 > 0) fill_coeff<PAIR>(Ct, stg, bb, nb, c.rp, r16 / 8, p, rank);
            } else if (cached) {
                fill_cache_keys<FMT, PAIR>(Kt, stg, nb, p, rank);
                if (!cache_keys_in_f16_range<FMT>(stg, nb, p)) atomicExch(err + 1, 1);
                // TAYLOR2: bf16 weights read by the Jensen MMA with Q K^T (stage s, free
                // since Q K^T of tile j - 2 completed; in a pair the even CTA holds the
                // weight rows, the odd CTA's rows stay zero); EXACT: fp32 steps read by the
                // softmax, in a ring of 4 like the tile info
                if (JENSEN == KV_JENSEN_TAYLOR2) {
                    if (rank == 0) fill_weights<FMT, JENSEN>(sm + M::w + s * kWBytes, stg, nb, p, jcoef, G::kWR);
                } else if (JENSEN == KV_JENSEN_EXACT) {
                    fill_weights<FMT, JENSEN>(sm + M::w + (j & 3) * kExactW, stg, nb, p, jcoef, G::kWR);
                } else if (JENSEN == KV_JENSEN_ISOTROPIC) {
                    fill_weights<FMT, JENSEN>(nullptr, stg, nb, p, jcoef, G::kWR, inf.ss2);
                }
            } else {
                if (!fill_current_keys<PAIR>(Kt, Kcur, row0, cvalid, p, rank)) atomicExch(err + 1, 1);
            }
            fence_proxy_async();
            // publish tile j on K_FULL[s] only after the softmax has finished tile j - 2
            // (its P_FULL[s]): the softmax then has passed its K_FULL[s] wait for tile j - 2,
            // so that wait can never find the barrier two phases ahead
            if (j >= 2) {
                const bool okp = mbar_wait(bar(BAR_P_FULL + s), ((j - 2) >> 1) & 1, &abort_flag, err, 11);
                if (!__all_sync(0xffffffffu, okp)) break;
            }
            mbar_arrive(bar(BAR_K_FULL + s));
            // values: the V_hat stage is free once P V of tile j - 2 completed; Q K^T and
            // the softmax of this tile proceed meanwhile
            const bool ok2 = j < 2 || mbar_wait(bar(BAR_V_EMPTY + s), ((j - 2) >> 1) & 1, &abort_flag, err, 2);
            if (!__all_sync(0xffffffffu, ok2)) break;
            unsigned char* Vt = sm + M::v + s * M::kTileV;
            if (cached) fill_cache_values<FMT, PAIR>(Vt, stg, bb, nb, pw, lane, rank);
            else fill_current_values<PAIR>(Vt, Vcur, row0, cvalid, p, rank);
            fence_proxy_async();
            mbar_arrive(bar(BAR_V_FULL + s));
            if (cached) {
                // staging slot s is consumed; thread 0 refills it with tile j + 2 once
                // every producer has arrived (a bounded wait, like all others)
                mbar_arrive(bar(BAR_STG_EMPTY + s));
                if (p == 0 && j + 2 < T && tile_of(j + 2) < n_cache_tiles &&
                    mbar_wait(bar(BAR_STG_EMPTY + s), (j >> 1) & 1, &abort_flag, err, 10)) {
                    stage_copy(j + 2);
                    issued = j + 3;
                }
            }
        }
        if (p == 0) {
            // copies still in flight after an abort land (bounded wait) before the CTA exits
            for (int jj = j; jj < issued; ++jj) {
                if (tile_of(jj) >= n_cache_tiles) continue;
                const long long t0c = clock64();
                while (!mbar_try_wait(bar(BAR_STG_FULL + (jj & 1)), (jj >> 1) & 1) && clock64() - t0c < 100000000LL) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int i = tid;                          // query row = TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const float c1 = tau * kLog2e;
        // ISOTROPIC: (tau^2 / 24) log2(e) |q|^2 / d of this row, times a block's sum of s_c^2
        float iso_c = 0.0f;
        if (JENSEN == KV_JENSEN_ISOTROPIC) {
            float qn2 = 0.0f;
            for (int ch = 0; ch < 16; ++ch) {
                const uint4 qv = q0 + i < n_q ? __ldg(Qg + (long long)(q0 + i) * (kD / 8) + ch) : make_uint4(0, 0, 0, 0);
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = __uint_as_float(qw[k] << 16), hi = __uint_as_float(qw[k] & 0xFFFF0000u);
                    qn2 = fmaf(lo, lo, fmaf(hi, hi, qn2));
                }
            }
            iso_c = tau * tau * (1.0f / 24.0f) * kLog2e * qn2 * (1.0f / kD);
        }
        float m_ref = -INFINITY, l_sum = 0.0f;
        float x[32];
        for (int j = 0; j < T; ++j) {
            const int s = j & 1;
            const bool ok0 = mbar_wait(bar(BAR_K_FULL + s), (j >> 1) & 1, &abort_flag, err, 4);
            if (!__all_sync(0xffffffffu, ok0)) break;
            const TileInfo info = infos[j & 3];
            // (failure tests: with `stall` the first wait targets a barrier nothing arrives
            // on, with a short limit, so the bounded-wait abort path runs)
            const bool ok1 = stall && j == 0 ? mbar_wait(bar(BAR_NEVER), 0, &abort_flag, err, 12, 1LL << 21)
                                             : mbar_wait(bar(BAR_S_FULL + s), (j >> 1) & 1, &abort_flag, err, 5);
            if (!__all_sync(0xffffffffu, ok1)) break;
            fence_after();
            float dl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (kCb) {
                if (JENSEN != KV_JENSEN_OFF && info.quantised) dl[0] = dl[1] = dl[2] = dl[3] = jrow;
            } else if (info.quantised) {
                if (JENSEN == KV_JENSEN_TAYLOR2) {
                    float dv[8];
                    tmem_ld8(tmem + lane_addr + kColD + G::kJN * s, dv);
#pragma unroll
                    for (int g = 0; g < 4; ++g) dl[g] = dv[g] + dv[4 + g];
                } else if (JENSEN == KV_JENSEN_EXACT) {
                    const float* SK = reinterpret_cast<const float*>(sm + M::w + (j & 3) * kExactW);
                    const float jt = 0.5f * tau;
#pragma unroll 2
                    for (int ch = 0; ch < 16; ++ch) {
                        const uint4 qv = *reinterpret_cast<const uint4*>(sm + M::q2h + sw_off(i, ch));
                        const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                        // per channel, the 4 blocks' arguments of the warp's 32 rows: when none
                        // reaches 1/2 the series alone, without branches (the same value the
                        // per-argument function gives); large-step channels take that function
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float qf = __uint_as_float(k & 1 ? (qw[k >> 1] & 0xFFFF0000u) : (qw[k >> 1] << 16));
                            float xa[4];
#pragma unroll
                            for (int g = 0; g < 4; ++g) xa[g] = fabsf(jt * qf * SK[g * kD + 8 * ch + k]);
                            const float xm = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
                            if (__any_sync(0xffffffffu, !(xm < 0.5f))) {
#pragma unroll
                                for (int g = 0; g < 4; ++g) dl[g] += log_sinhc(xa[g]);
                            } else {
#pragma unroll
                                for (int g = 0; g < 4; ++g) dl[g] += log_sinhc_series(xa[g]);
                            }
                        }
                    }
#pragma unroll
                    for (int g = 0; g < 4; ++g) dl[g] *= kLog2e;
                } else if (JENSEN == KV_JENSEN_ISOTROPIC) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) dl[g] = iso_c * (info.ss2[g][0] + info.ss2[g][1]);
                }
            }
            // pass 1: the tile's maximum of the corrected logits (log2 units)
            float mt = -INFINITY;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int nv = info.nvalid[g];
                tmem_ld32(tmem + lane_addr + kColS + s * kN + 32 * g, x);
                float mx = -INFINITY;
                if (nv == 32) {
#pragma unroll
                    for (int k = 0; k < 32; k += 2) mx = fmax3(mx, x[k], x[k + 1]);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) mx = fmaxf(mx, k < nv ? x[k] : -INFINITY);
                }
                if (nv > 0) mt = fmaxf(mt, fmaf(mx, c1, -dl[g]));
            }
            const float m_new = fmaxf(m_ref, mt);
            // rescale only when the max grows by more than 2^15: p <= 2^15 stays inside
            // fp16 (max 65504) and its relative precision does not depend on the scale
            const bool grow = m_new > m_ref + 15.0f;      // also true for the first finite max
            // O is rescaled in TMEM when any row of the warp needs it, after P V of
            // tile j - 1 has completed; tcgen05.ld/st are warp-collective, so the whole
            // warp takes the branch (alpha = 1 for rows whose running max did not move).
            const bool resc = grow && j > 0;
            const float alpha = resc ? ex2(m_ref - m_new) : 1.0f;
            if (__any_sync(0xffffffffu, resc)) {
                const bool ok2 = mbar_wait(bar(BAR_O_DONE), (j - 1) & 1, &abort_flag, err, 6);
                if (!__all_sync(0xffffffffu, ok2)) break;
                fence_after();
                float ob[32];
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    tmem_ld32(tmem + lane_addr + kColO + 32 * g, ob);
#pragma unroll
                    for (int k = 0; k < 32; ++k) ob[k] *= alpha;
                    tmem_st32(tmem + lane_addr + kColO + 32 * g, ob);
                }
            }
            l_sum *= alpha;
            if (grow) m_ref = m_new;
            const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
            // pass 2: p = 2^(S c1 - (m + delta_g)), summed in fp32, stored as fp16 over the
            // S columns already read (group g's 16 columns of P land in columns 16 g ..)
            float psum = 0.0f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int nv = info.nvalid[g];
                tmem_ld32(tmem + lane_addr + kColS + s * kN + 32 * g, x);
                const float bg = m_use + dl[g];
                uint32_t u[16];
                if (nv == 32) {
                    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        float e0, e1;
                        fma2(e0, e1, x[2 * k], x[2 * k + 1], c1, c1, -bg, -bg);
                        const float p0 = ex2(e0), p1 = ex2(e1);
                        add2(a0, a1, a0, a1, p0, p1);
                        u[k] = pack_f16(p0, p1);
                    }
                    psum += a0 + a1;
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float p0 = 2 * k < nv ? ex2(fmaf(x[2 * k], c1, -bg)) : 0.0f;
                        const float p1 = 2 * k + 1 < nv ? ex2(fmaf(x[2 * k + 1], c1, -bg)) : 0.0f;
                        psum += p0 + p1;
                        u[k] = pack_f16(p0, p1);
                    }
                }
                tmem_st16(tmem + lane_addr + kColS + s * kN + 16 * g, u);
            }
            l_sum += psum;
            tmem_wait_st();
            fence_before();
            mbar_arrive(bar(BAR_P_FULL + s));
        }
        // ---- epilogue
        const int qi = q0 + i;
        const long long orow = ((long long)b * Hq + hq) * n_q + qi;
        // O is final once every MMA of the CTA has completed (MMA_DONE, committed once
        // after the last P V).  A parity wait on O_DONE for the last tile would be
        // ambiguous here: the tile before it may not have completed either, and a
        // barrier two phases behind shows the awaited parity as done.
        bool have = T > 0 && !abort_flag;
        if (have) have = mbar_wait(bar(BAR_MMA_DONE), 0, &abort_flag, err, 7);
        have = __all_sync(0xffffffffu, have);
        fence_after();
        const float inv = l_sum > 0.0f ? 1.0f / l_sum : 0.0f;
        const long long rows = (long long)c.B * Hq * n_q;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            float ob[32];
            __syncwarp();
            if (have) {
                tmem_ld32(tmem + lane_addr + kColO + 32 * g, ob);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) ob[k] = 0.0f;
            }
            if (qi < n_q) {
                if (n_splits == 1) {
                    if (out_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + orow * kD + 32 * g);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(ob[4 * k] * inv, ob[4 * k + 1] * inv, ob[4 * k + 2] * inv,
                                                 ob[4 * k + 3] * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + orow * kD + 32 * g);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(pack_bf16(ob[8 * k] * inv, ob[8 * k + 1] * inv),
                                                pack_bf16(ob[8 * k + 2] * inv, ob[8 * k + 3] * inv),
                                                pack_bf16(ob[8 * k + 4] * inv, ob[8 * k + 5] * inv),
                                                pack_bf16(ob[8 * k + 6] * inv, ob[8 * k + 7] * inv));
                    }
                } else {
                    float4* dst = reinterpret_cast<float4*>(ws_o + ((long long)split * rows + orow) * kD + 32 * g);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(ob[4 * k] * inv, ob[4 * k + 1] * inv, ob[4 * k + 2] * inv,
                                             ob[4 * k + 3] * inv);
                }
            }
        }
        if (qi < n_q) {
            if (n_splits == 1) {
                if (lse) lse[orow] = l_sum > 0.0f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
            } else {
                ws_ml[(long long)split * rows + orow] = make_float2(l_sum > 0.0f ? m_ref * kLn2 : -INFINITY, l_sum);
            }
        }
        __syncwarp();
    }
    fence_before();
    __syncthreads();
    // a pair: neither CTA frees its tensor memory or exits (its shared memory) while the
    // other may still signal it; the even CTA's MMAs have all completed (MMA_DONE)
    if (PAIR) cluster_sync();
    if (warp == kMmaWarp) {
        fence_after();
        if (PAIR) tmem_dealloc2(tmem, kTmemCols);
        else tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------- operand dump -----
// Debug view of the kernel's own operands: the fp16 K_hat and V_hat that the
// expansion routines above (the same functions the attention kernel's producers
// run) build from one staged cache tile, written un-swizzled in block-slot order
// as fp16 [B][Hkv][32 n_blocks][d] (V_hat transposed back to token rows).  One CTA
// of 256 threads per (tile, kv head, batch); rows of missing blocks are not written.
template <int FMT>
struct DumpSmem {
    static constexpr int k = 0;
    static constexpr int v = k + kTile;
    static constexpr int cent = v + kTile;
    static constexpr int stg = cent + kCentBytes;
    static constexpr int total = stg + 4 * max_block_bytes<FMT>() + 1024;
};

template <int FMT>
__global__ void __launch_bounds__(kProd)
tc_operands_kernel(DevCache c, __half* __restrict__ Kout, __half* __restrict__ Vout) {
    using M = DumpSmem<FMT>;
    constexpr bool kCb = FMT == FMT_CB2;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int p = threadIdx.x, pw = p >> 5, lane = p & 31;
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int seg = seg_of<FMT>();
    const int nblk = c.n_blocks[seg];
    const int nb = min(4, nblk - tile * 4);
    if (nb <= 0) return;
    const int bb = kCb ? (int)c.block_bytes[seg] : max_block_bytes<FMT>();
    // stage the tile's blocks (plain 16-byte copies: the staging method is not under test)
    const uint4* src = reinterpret_cast<const uint4*>(block_ptr(c, b, h, seg, tile * 4));
    uint4* dst = reinterpret_cast<uint4*>(sm + M::stg);
    for (int e = p; e < nb * bb / 16; e += kProd) dst[e] = src[e];
    if (kCb) fill_centroid_tables(reinterpret_cast<uint32_t*>(sm + M::cent),
                                  c.centroids + ((long long)b * c.Hkv + h) * kD * 4, p);
    __syncthreads();
    // keys first, then values (the value routine rescales the staged steps in place)
    if (kCb) fill_cb_keys<false>(sm + M::k, sm + M::stg, bb, nb, reinterpret_cast<const uint32_t*>(sm + M::cent), p, 0);
    else fill_cache_keys<FMT, false>(sm + M::k, sm + M::stg, nb, p, 0);
    __syncthreads();
    fill_cache_values<FMT, false>(sm + M::v, sm + M::stg, bb, nb, pw, lane, 0);
    __syncthreads();
    const long long row0 = ((long long)b * c.Hkv + h) * (long long)nblk * kBlockTokens + (long long)tile * kN;
    for (int e = p; e < nb * kBlockTokens * (kD / 8); e += kProd) {
        const int row = e / (kD / 8), ch = e % (kD / 8);
        *reinterpret_cast<uint4*>(Kout + (row0 + row) * kD + 8 * ch) =
            *reinterpret_cast<const uint4*>(sm + M::k + sw_off(row, ch));
    }
    for (int e = p; e < nb * kBlockTokens * kD; e += kProd) {
        const int key = e / kD, ch = e % kD;
        Vout[(row0 + key) * kD + ch] =
            *reinterpret_cast<const __half*>(sm + M::v + sw_off(ch, key >> 3) + 2 * (key & 7));
    }
}

template <int FMT>
kv_status launch_tc_operands_t(const DevCache& c, void* Kout, void* Vout, cudaStream_t st) {
    constexpr int kSmem = DumpSmem<FMT>::total;
    const kv_status sa = set_smem_limit(reinterpret_cast<const void*>(tc_operands_kernel<FMT>), kSmem,
                                        "tc_operands_kernel");
    if (sa != KV_OK) return sa;
    const int seg = seg_of<FMT>();
    const int tiles = (c.n_blocks[seg] + 3) / 4;
    if (tiles == 0) return KV_OK;
    tc_operands_kernel<FMT><<<dim3(tiles, c.Hkv, c.B), kProd, kSmem, st>>>(c, static_cast<__half*>(Kout),
                                                                          static_cast<__half*>(Vout));
    return check_launch("tc_operands_kernel");
}

int g_num_sms = 0;

int num_sms() {
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

template <int FMT, int JENSEN, bool PAIR>
kv_status launch_tc_p(const DevCache& c, const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                      float tau, int r16, int n_splits, void* out, int out_f32, float* lse, float* ws_o, float2* ws_ml,
                      int* err, cudaStream_t st) {
    constexpr int kSmem = Smem<FMT, PAIR>::total;
    auto kern = attn_tc_kernel<FMT, JENSEN, PAIR>;
    const kv_status sa = set_smem_limit(reinterpret_cast<const void*>(kern), kSmem, "attn_tc_kernel");
    if (sa != KV_OK) return sa;
    const int n_qt = (n_q + kM - 1) / kM;
    const int stall = getenv("BITKV_TEST_NEVER_ARRIVE") != nullptr ? 1 : 0;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(Q);
    const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(Kc);
    const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(Vc);
    if (!PAIR) {
        dim3 grid(n_qt * n_splits, Hq, c.B);
        kern<<<grid, kThreads, kSmem, st>>>(q, kc, vc, n_q, n_cur, Hq, c, tau, r16, n_splits, out, out_f32, lse, ws_o,
                                            ws_ml, err, stall);
        return check_launch("attn_tc_kernel");
    }
    // pairs of query tiles in 2-CTA clusters
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((n_qt + 1) / 2) * n_splits, Hq, c.B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q, kc, vc, n_q, n_cur, Hq, c, tau, r16, n_splits, out, out_f32,
                                             lse, ws_o, ws_ml, err, stall);
    if (e != cudaSuccess) return set_error(KV_ERR_CUDA, "attn_tc_kernel (CTA pairs): %s", cudaGetErrorString(e));
    return check_launch("attn_tc_kernel");
}

template <int FMT, int JENSEN>
kv_status launch_tc_t(const DevCache& c, const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                      float tau, int r16, int n_splits, void* out, int out_f32, float* lse, float* ws_o, float2* ws_ml,
                      int* err, bool pair, cudaStream_t st) {
    if (pair)
        return launch_tc_p<FMT, JENSEN, true>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, r16, n_splits, out, out_f32, lse,
                                              ws_o, ws_ml, err, st);
    return launch_tc_p<FMT, JENSEN, false>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, r16, n_splits, out, out_f32, lse, ws_o,
                                           ws_ml, err, st);
}

}  // namespace

bool tc_supported(const kv_cache* cache, kv_dtype dt, int n_q, int Hq, const char** why) {
    const kv_layout& L = cache->layout;
    (void)Hq;
    if (dt != KV_BF16) { *why = "needs bf16 I/O"; return false; }
    if (L.d != kD) { *why = "needs head dim 128"; return false; }
    if (L.kind != KV_UNIFORM2 && L.kind != KV_UNIFORM4 && L.kind != KV_CODEBOOK2) {
        *why = "needs a UNIFORM2, UNIFORM4 or CODEBOOK2 cache";
        return false;
    }
    if (n_q < 16) { *why = "needs at least 16 queries"; return false; }
    return true;
}

int tc_auto_splits(const kv_cache* cache, int n_q, int n_cur, int Hq, bool pair) {
    const kv_layout& L = cache->layout;
    const int seg = L.kind == KV_UNIFORM4 ? KV_SEG_INT4 : KV_SEG_INT2;
    const int tiles = (cache->n_blocks[seg] + 3) / 4 + (n_cur + kN - 1) / kN;
    const int n_qt = (n_q + kM - 1) / kM;
    const long long ctas = (long long)L.B * Hq * (pair ? 2 * ((n_qt + 1) / 2) : n_qt);
    // pipeline fill per CTA, in tiles: longer for a pair, whose halves meet through the cluster
    const double fill = pair ? 6.0 : 3.0;
    const int sms = num_sms();
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 8; ++s) {
        if (s > 1 && tiles / s < 6) break;
        const double waves = (double)((ctas * s + sms - 1) / sms);
        const double cost = waves * ((double)tiles / s + fill);
        if (cost < best_cost * 0.97) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

size_t tc_workspace(const kv_cache* cache, int n_q, int Hq, int n_splits) {
    size_t ws = kStatusBytes;
    if (n_splits > 1) {
        const long long rows = (long long)cache->layout.B * Hq * n_q;
        ws += (size_t)n_splits * rows * (kD * sizeof(float) + sizeof(float2));
    }
    return ws;
}

kv_status launch_attn_tc(const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                         const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out, int out_f32,
                         float* lse, void* ws, bool pair, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    int* err = static_cast<int*>(ws);
    float* ws_o = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kStatusBytes);
    const long long rows = (long long)c.B * Hq * n_q;
    float2* ws_ml = reinterpret_cast<float2*>(ws_o + (n_splits > 1 ? (long long)n_splits * rows * kD : 0));
    kv_status s = clear_device(ws, kStatusBytes, st, "attn_tc_kernel");
    if (s != KV_OK) return s;
#define BITKV_TC(FMT)                                                                                         \
    switch (jensen) {                                                                                         \
        case KV_JENSEN_TAYLOR2:                                                                               \
            s = launch_tc_t<FMT, KV_JENSEN_TAYLOR2>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, 0, n_splits, out,      \
                                                    out_f32, lse, ws_o, ws_ml, err, pair, st);                      \
            break;                                                                                            \
        case KV_JENSEN_EXACT:                                                                                 \
            s = launch_tc_t<FMT, KV_JENSEN_EXACT>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, 0, n_splits, out, out_f32, \
                                                  lse, ws_o, ws_ml, err, pair, st);                                 \
            break;                                                                                            \
        case KV_JENSEN_ISOTROPIC:                                                                             \
            s = launch_tc_t<FMT, KV_JENSEN_ISOTROPIC>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, 0, n_splits, out,    \
                                                      out_f32, lse, ws_o, ws_ml, err, pair, st);                    \
            break;                                                                                            \
        default:                                                                                              \
            s = launch_tc_t<FMT, KV_JENSEN_OFF>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, 0, n_splits, out, out_f32,   \
                                                lse, ws_o, ws_ml, err, pair, st);                                   \
    }
    if (c.kind == KV_CODEBOOK2) {
        // codebook keys carry no step sizes: their Jensen term needs the residual variances
        const int r16 = psac ? (c.r + 15) / 16 * 16 : 0;
        const int jm = c.resid_var ? jensen : KV_JENSEN_OFF;
        if (jm == KV_JENSEN_TAYLOR2)
            s = launch_tc_t<FMT_CB2, KV_JENSEN_TAYLOR2>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, r16, n_splits, out, out_f32,
                                                        lse, ws_o, ws_ml, err, pair, st);
        else if (jm == KV_JENSEN_ISOTROPIC)
            s = launch_tc_t<FMT_CB2, KV_JENSEN_ISOTROPIC>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, r16, n_splits, out,
                                                          out_f32, lse, ws_o, ws_ml, err, pair, st);
        else
            s = launch_tc_t<FMT_CB2, KV_JENSEN_OFF>(c, Q, Kc, Vc, n_q, n_cur, Hq, tau, r16, n_splits, out, out_f32,
                                                    lse, ws_o, ws_ml, err, pair, st);
    } else if (c.kind == KV_UNIFORM4) {
        if (c.meta16) {
            BITKV_TC(FMT_INT4H)
        } else {
            BITKV_TC(FMT_INT4)
        }
    } else if (c.meta16) {
        BITKV_TC(FMT_INT2H)
    } else {
        BITKV_TC(FMT_INT2)
    }
#undef BITKV_TC
    if (s != KV_OK) return s;
    if (n_splits == 1) return KV_OK;
    return launch_lse_merge(KV_BF16, ws_o, ws_ml, n_splits, rows, kD, out, out_f32, lse, st);
}

kv_status launch_tc_operands(const kv_cache* cache, void* Kout, void* Vout, cudaStream_t st) {
    const DevCache c = make_dev_cache(cache);
    if (c.d != kD) return set_error(KV_ERR_UNSUPPORTED, "tensor-core operands: needs head dim 128");
    if (c.kind == KV_CODEBOOK2) return launch_tc_operands_t<FMT_CB2>(c, Kout, Vout, st);
    if (c.kind == KV_UNIFORM4)
        return c.meta16 ? launch_tc_operands_t<FMT_INT4H>(c, Kout, Vout, st)
                        : launch_tc_operands_t<FMT_INT4>(c, Kout, Vout, st);
    if (c.kind == KV_UNIFORM2)
        return c.meta16 ? launch_tc_operands_t<FMT_INT2H>(c, Kout, Vout, st)
                        : launch_tc_operands_t<FMT_INT2>(c, Kout, Vout, st);
    return set_error(KV_ERR_UNSUPPORTED, "tensor-core operands: needs a UNIFORM2, UNIFORM4 or CODEBOOK2 cache");
}

}  // namespace bitkv
