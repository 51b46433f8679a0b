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
//   warps 0-3  softmax: thread i owns query row i = TMEM lane i.  Loads the S
//              row from TMEM, applies scale, Jensen delta and the key mask,
//              keeps a lazily rescaled running max (O is rescaled in TMEM only
//              when the max grows by more than 2^8), writes P (fp16) to smem.
//   warps 4-7  producers: thread 0 bulk-copies (TMA engine) each packed cache
//              tile -- 4 contiguous blocks -- into a double-buffered staging
//              area two tiles ahead; all 128 threads dequantise the staged
//              tile into K_hat [128 keys x 128] (bf16, single buffer: free once
//              Q K_hat^T of the tile completes) and V_hat^T [128 channels x 128
//              keys] (fp16, double buffer), 128-byte-swizzled K-major; a
//              current-chunk tile is read from global memory and transposed.
//   warp 8     TMEM owner; lane 0 issues S = Q K_hat^T (bf16) and O += P V_hat (fp16).
// TMEM: S double buffer (columns 0-255), O (256-383).  Every wait is bounded;
// every warp-collective tcgen05 load/store runs with the whole warp converged.
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
constexpr int kThreads = 288;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_bf16(kM, kN);   // S = Q K_hat^T, bf16 operands
constexpr uint32_t kIdescPV = idesc_f16(kM, kD);    // O += P V_hat, fp16 operands
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory map (bytes from a 1024-aligned base)
constexpr int kTile = kM * kD * 2;          // 32 KB: one 16-bit 128 x 128 operand tile
constexpr int kStage = 4 * 6144;            // packed bytes of 4 INT4 blocks (INT2: 4 x 4096)
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTile;        // 1 buffer
constexpr int kVOff = kKOff + kTile;        // 2 stages
constexpr int kPOff = kVOff + 2 * kTile;
constexpr int kStgOff = kPOff + kTile;      // 2 staging slots of packed blocks
constexpr int kWOff = kStgOff + 2 * kStage; // 2 stages x 4 groups x 128 floats (Jensen weights)
constexpr int kInfoOff = kWOff + 2 * 4 * kD * 4;
constexpr int kStgLenOff = kInfoOff + 2 * 32;   // [2][4] valid lengths of the staged blocks
constexpr int kBarOff = kStgLenOff + 2 * 16;
constexpr int kNumBars = 13;
constexpr int kSlotOff = kBarOff + kNumBars * 8;
constexpr int kSmemUsed = kSlotOff + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack

enum {
    BAR_KV_FULL = 0,   // [2] producers -> MMA/softmax: K_hat, V_hat[s], weights[s], info[s] ready
    BAR_V_EMPTY = 2,   // [2] PV of the stage's tile completed
    BAR_S_FULL = 4,    // [2] S = Q K_hat^T of the tile in TMEM
    BAR_P_FULL = 6,    // softmax -> MMA: P written
    BAR_O_DONE = 7,    // PV completed
    BAR_K_EMPTY = 8,   // Q K_hat^T completed (K_hat may be overwritten)
    BAR_STG_FULL = 9,  // [2] staging slot filled by the bulk copy
    BAR_STG_EMPTY = 11,  // [2] all producers finished reading the staging slot
};

struct TileInfo {
    int nvalid[4];
    int quantised;
    int pad[3];
};

// Byte offset of 16-byte chunk `ch` (0..15) of row `row` in a 128-row x 128-column
// 16-bit tile stored as two 64-column, 128-byte-swizzled K-major halves.
__device__ __forceinline__ uint32_t sw_off(int row, int ch) {
    return (uint32_t)((ch >> 3) * (kM * 128) + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// Dequantise 8 codes and pack them as bf16 (keys, F16OUT = false) or fp16 (values).
template <bool F16OUT>
__device__ __forceinline__ uint4 dq8_pack(const uint32_t codes[8], const float s[8], const float z[8]) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = dequant(codes[k], s[k], z[k]);
    uint4 r;
    if (F16OUT) {
        r.x = pack_f16(v[0], v[1]);
        r.y = pack_f16(v[2], v[3]);
        r.z = pack_f16(v[4], v[5]);
        r.w = pack_f16(v[6], v[7]);
    } else {
        r.x = pack_bf16(v[0], v[1]);
        r.y = pack_bf16(v[2], v[3]);
        r.z = pack_bf16(v[4], v[5]);
        r.w = pack_bf16(v[6], v[7]);
    }
    return r;
}

// ------------------------------------------------------------- producers ----
// A staged cache tile: 4 consecutive blocks (the missing ones of a short last
// tile count as empty) in staging slot `stage`, their valid lengths in stg_len.
struct StagedTile {
    const unsigned char* stg;
    const int* len;
    int nb;   // blocks present
};

// Values: thread p dequantises channel p of all 128 keys into V_hat^T[stage] and
// records the tile's key-validity info.
template <int BITS>
__device__ void fill_cache_values(unsigned char* sm, int stage, const StagedTile& st, int p) {
    const IntBlockOffsets o = int_offsets(kD, BITS);
    constexpr int kBlockBytes = 8 * kD * BITS + 16 * kD;
    unsigned char* Vt = sm + kVOff + stage * kTile;
    TileInfo* info = reinterpret_cast<TileInfo*>(sm + kInfoOff) + stage;
    if (p < 4) info->nvalid[p] = p < st.nb ? st.len[p] : 0;
    if (p == 0) info->quantised = 1;
    const int cc = p;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        if (q < st.nb) {
            const unsigned char* blk = st.stg + q * kBlockBytes;
            const uint32_t* vc = reinterpret_cast<const uint32_t*>(blk + o.vc) + cc * BITS;
            const float4* vm = reinterpret_cast<const float4*>(blk + o.vm) + (cc >> 5) * 16;  // 32 float2
            uint32_t wv[BITS];
#pragma unroll
            for (int k = 0; k < BITS; ++k) wv[k] = vc[k];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float vs[8], vz[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 v = vm[kk * 4 + k];
                    vs[2 * k] = v.x;
                    vz[2 * k] = v.y;
                    vs[2 * k + 1] = v.z;
                    vz[2 * k + 1] = v.w;
                }
                uint32_t codes[8];
                if (BITS == 2) {
                    const uint32_t w = wv[kk >> 1] >> (16 * (kk & 1));
#pragma unroll
                    for (int k = 0; k < 8; ++k) codes[k] = (w >> (2 * k)) & 3u;
                } else {
                    const uint32_t w = wv[kk];
#pragma unroll
                    for (int k = 0; k < 8; ++k) codes[k] = (w >> (4 * k)) & 15u;
                }
                *reinterpret_cast<uint4*>(Vt + sw_off(cc, 4 * q + kk)) = dq8_pack<true>(codes, vs, vz);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                *reinterpret_cast<uint4*>(Vt + sw_off(cc, 4 * q + kk)) = make_uint4(0, 0, 0, 0);
        }
    }
}

// Keys: thread p dequantises channels 8jc..8jc+7 of keys r0, r0+8, ... into the
// single K_hat buffer and stores the Jensen weights of its channels.
template <int BITS>
__device__ void fill_cache_keys(unsigned char* sm, int stage, const StagedTile& st, int p, int jensen) {
    const IntBlockOffsets o = int_offsets(kD, BITS);
    constexpr int kBlockBytes = 8 * kD * BITS + 16 * kD;
    constexpr int kWordsPerKey = kD * BITS / 32;
    unsigned char* Kt = sm + kKOff;
    float* W = reinterpret_cast<float*>(sm + kWOff) + stage * 4 * kD;
    const int jc = p & 15, r0 = p >> 4;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        const bool exists = q < st.nb;
        const unsigned char* blk = st.stg + q * kBlockBytes;
        float s[8], z[8];
        if (exists) {
            const float4* km = reinterpret_cast<const float4*>(blk + o.km) + jc * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = km[k];
                s[2 * k] = v.x;
                z[2 * k] = v.y;
                s[2 * k + 1] = v.z;
                z[2 * k + 1] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) s[k] = z[k] = 0.0f;
        }
        if (r0 == 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                W[q * kD + jc * 8 + k] = jensen == KV_JENSEN_EXACT ? s[k] : s[k] * s[k];
        }
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(blk + o.kc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = r0 + 8 * i;
            const int row = 32 * q + t;
            uint4 pk = make_uint4(0, 0, 0, 0);
            if (exists) {
                uint32_t codes[8];
                if (BITS == 2) {
                    const uint32_t w = kc[t * kWordsPerKey + (jc >> 1)] >> (16 * (jc & 1));
#pragma unroll
                    for (int k = 0; k < 8; ++k) codes[k] = (w >> (2 * k)) & 3u;
                } else {
                    const uint32_t w = kc[t * kWordsPerKey + jc];
#pragma unroll
                    for (int k = 0; k < 8; ++k) codes[k] = (w >> (4 * k)) & 15u;
                }
                pk = dq8_pack<false>(codes, s, z);
            }
            *reinterpret_cast<uint4*>(Kt + sw_off(row, jc)) = pk;
        }
    }
}

// Two bf16 values (half `hf` of two words) converted to an fp16 pair.
__device__ __forceinline__ uint32_t f16_pair_from_bf16(uint32_t lo_word, uint32_t hi_word, int hf) {
    const float lo = __uint_as_float(hf ? (lo_word & 0xFFFF0000u) : (lo_word << 16));
    const float hi = __uint_as_float(hf ? (hi_word & 0xFFFF0000u) : (hi_word << 16));
    return pack_f16(lo, hi);
}

// Current-chunk tile (unquantised bf16): values transposed to fp16 V_hat^T, and
// the key-validity info.
__device__ void fill_current_values(unsigned char* sm, int stage, const __nv_bfloat16* Vcur, long long row0,
                                    int valid, int p) {
    unsigned char* Vt = sm + kVOff + stage * kTile;
    TileInfo* info = reinterpret_cast<TileInfo*>(sm + kInfoOff) + stage;
    if (p < 4) info->nvalid[p] = min(32, max(0, valid - 32 * p));
    if (p == 0) info->quantised = 0;
    const uint4* Vg = reinterpret_cast<const uint4*>(Vcur + row0 * kD);
    uint32_t x[2][8][4];                 // both 8x8 blocks' loads in flight before any store
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
        const int bi = p + 128 * rep;
        const int kc8 = bi >> 4, cch = bi & 15;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int key = 8 * kc8 + k;
            const uint4 v = key < valid ? __ldg(Vg + key * (kD / 8) + cch) : make_uint4(0, 0, 0, 0);
            x[rep][k][0] = v.x;
            x[rep][k][1] = v.y;
            x[rep][k][2] = v.z;
            x[rep][k][3] = v.w;
        }
    }
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
        const int bi = p + 128 * rep;
        const int kc8 = bi >> 4, cch = bi & 15;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // channel 8cch+i: element i of every key row (word i/2, half i&1)
            const int wi = i >> 1, hf = i & 1;
            uint4 y;
            y.x = f16_pair_from_bf16(x[rep][0][wi], x[rep][1][wi], hf);
            y.y = f16_pair_from_bf16(x[rep][2][wi], x[rep][3][wi], hf);
            y.z = f16_pair_from_bf16(x[rep][4][wi], x[rep][5][wi], hf);
            y.w = f16_pair_from_bf16(x[rep][6][wi], x[rep][7][wi], hf);
            *reinterpret_cast<uint4*>(Vt + sw_off(8 * cch + i, kc8)) = y;
        }
    }
}

// Current-chunk keys: bf16 rows copied into the swizzled K_hat buffer.
__device__ void fill_current_keys(unsigned char* sm, const __nv_bfloat16* Kcur, long long row0, int valid, int p) {
    unsigned char* Kt = sm + kKOff;
    const int jc = p & 15, r0 = p >> 4;
    const uint4* Kg = reinterpret_cast<const uint4*>(Kcur + row0 * kD);
    uint4 kv[16];                        // all loads in flight before the first store
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int row = r0 + 8 * i;
        kv[i] = row < valid ? __ldg(Kg + row * (kD / 8) + jc) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) *reinterpret_cast<uint4*>(Kt + sw_off(r0 + 8 * i, jc)) = kv[i];
}

// --------------------------------------------------------------- kernel -----
template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kcur,
               const __nv_bfloat16* __restrict__ Vcur, int n_q, int n_cur, int Hq, DevCache c, float tau, int jensen,
               int n_splits, void* __restrict__ out, int out_f32, float* __restrict__ lse, float* __restrict__ ws_o,
               float2* __restrict__ ws_ml, int* __restrict__ err) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ volatile int abort_flag;
    unsigned char* sm =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n_qt = (n_q + kM - 1) / kM;
    const int qt = blockIdx.x % n_qt, split = blockIdx.x / n_qt;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int h = hq / (Hq / c.Hkv);
    const int q0 = qt * kM;
    const int seg = BITS == 4 ? KV_SEG_INT4 : KV_SEG_INT2;
    const int n_cache_tiles = (c.n_blocks[seg] + 3) / 4;
    const int n_tiles = n_cache_tiles + (n_cur + kN - 1) / kN;
    // split s takes tiles s, s + n_splits, ...: every split gets an even share of
    // cache and current-chunk tiles, and its cache tiles still come first.
    const int T = split < n_tiles ? (n_tiles - split + n_splits - 1) / n_splits : 0;
    auto tile_of = [&](int j) { return split + j * n_splits; };
    auto bar = [&](int i) { return sbase + kBarOff + 8 * i; };

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(bar(BAR_KV_FULL + 0), 128);
        mbar_init(bar(BAR_KV_FULL + 1), 128);
        mbar_init(bar(BAR_V_EMPTY + 0), 1);
        mbar_init(bar(BAR_V_EMPTY + 1), 1);
        mbar_init(bar(BAR_S_FULL + 0), 1);
        mbar_init(bar(BAR_S_FULL + 1), 1);
        mbar_init(bar(BAR_P_FULL), 128);
        mbar_init(bar(BAR_O_DONE), 1);
        mbar_init(bar(BAR_K_EMPTY), 1);
        mbar_init(bar(BAR_STG_FULL + 0), 1);
        mbar_init(bar(BAR_STG_FULL + 1), 1);
        mbar_init(bar(BAR_STG_EMPTY + 0), 128);
        mbar_init(bar(BAR_STG_EMPTY + 1), 128);
        mbar_fence_init();
    }
    if (warp == 8) tmem_alloc(sbase + kSlotOff, kTmemCols);

    // Q tile -> swizzled smem (rows beyond n_q are zero)
    if (tid < 256) {
        const uint4* Qg = reinterpret_cast<const uint4*>(Q + (((long long)b * Hq + hq) * n_q) * kD);
#pragma unroll 4
        for (int i = 0; i < 8; ++i) {
            const int e = tid + 256 * i;
            const int row = e >> 4, ch = e & 15;
            const uint4 v =
                (q0 + row < n_q) ? __ldg(Qg + (long long)(q0 + row) * (kD / 8) + ch) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sm + kQOff + sw_off(row, ch)) = v;
        }
    }
    fence_proxy_async();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kSlotOff);

    if (warp == 8) {
        // ---------------------------------------------------------- MMA issuer
        if ((tid & 31) == 0) {
            const uint32_t sQ = sbase + kQOff, sP = sbase + kPOff;
            auto issue_pv = [&](int jj) -> bool {
                if (!mbar_wait(bar(BAR_P_FULL), jj & 1, &abort_flag, err, 3)) return false;
                fence_after();
                const uint32_t sV = sbase + kVOff + (jj & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
                    mma_f16kind(tmem + 256, desc_sw128(sP + off), desc_sw128(sV + off), kIdescPV,
                                (jj > 0 || kk > 0));
                }
                mma_commit(bar(BAR_O_DONE));
                mma_commit(bar(BAR_V_EMPTY + (jj & 1)));
                return true;
            };
            bool ok = true;
            for (int j = 0; j < T && ok; ++j) {
                const int s = j & 1;
                if (!mbar_wait(bar(BAR_KV_FULL + s), (j >> 1) & 1, &abort_flag, err, 1)) break;
                fence_after();
                const uint32_t sK = sbase + kKOff;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
                    mma_f16kind(tmem + s * kN, desc_sw128(sQ + off), desc_sw128(sK + off), kIdescQK, kk > 0);
                }
                mma_commit(bar(BAR_S_FULL + s));
                mma_commit(bar(BAR_K_EMPTY));
                if (j > 0) ok = issue_pv(j - 1);
            }
            if (ok && T > 0 && !abort_flag) issue_pv(T - 1);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ----------------------------------------------------------- producers
        const int p = tid - 128;
        const int nblk = c.n_blocks[seg];
        int* stg_len = reinterpret_cast<int*>(sm + kStgLenOff);
        // Bulk-copy cache tile j (if it is one) into staging slot j & 1, with its
        // blocks' valid lengths; run by producer thread 0 two tiles ahead.
        auto stage_copy = [&](int j) {
            const int tile = tile_of(j);
            if (j >= T || tile >= n_cache_tiles) return;
            const int nb = min(4, nblk - tile * 4);
            for (int q = 0; q < 4; ++q)
                stg_len[(j & 1) * 4 + q] = q < nb ? c.blk_len[(long long)b * c.cap_total + c.seg_base[seg] + tile * 4 + q] : 0;
            const uint32_t bytes = (uint32_t)(nb * c.block_bytes[seg]);
            const uint32_t sbar = bar(BAR_STG_FULL + (j & 1));
            mbar_expect_tx(sbar, bytes);
            bulk_g2s(sbase + kStgOff + (j & 1) * kStage, block_ptr(c, b, h, seg, tile * 4), bytes, sbar);
        };
        if (p == 0) {
            stage_copy(0);
            stage_copy(1);
        }
        for (int j = 0; j < T; ++j) {
            const int s = j & 1;
            const int tile = tile_of(j);
            const bool cached = tile < n_cache_tiles;
            bool ok = true;
            if (j >= 2) ok = mbar_wait(bar(BAR_V_EMPTY + s), ((j - 2) >> 1) & 1, &abort_flag, err, 2);
            if (ok && cached) ok = mbar_wait(bar(BAR_STG_FULL + s), (j >> 1) & 1, &abort_flag, err, 9);
            if (!__all_sync(0xffffffffu, ok)) break;
            StagedTile st;
            st.stg = sm + kStgOff + s * kStage;
            st.len = stg_len + s * 4;
            st.nb = cached ? min(4, nblk - tile * 4) : 0;
            const int t0 = (tile - n_cache_tiles) * kN;
            const long long row0 = ((long long)b * c.Hkv + h) * n_cur + t0;
            // values first: they only need the V_hat stage, free since PV of tile j - 2
            if (cached) fill_cache_values<BITS>(sm, s, st, p);
            else fill_current_values(sm, s, Vcur, row0, min(kN, n_cur - t0), p);
            // keys: the single K_hat buffer is free once Q K_hat^T of tile j - 1 completed
            const bool ok2 = j == 0 || mbar_wait(bar(BAR_K_EMPTY), (j - 1) & 1, &abort_flag, err, 8);
            if (!__all_sync(0xffffffffu, ok2)) break;
            if (cached) fill_cache_keys<BITS>(sm, s, st, p, jensen);
            else fill_current_keys(sm, Kcur, row0, min(kN, n_cur - t0), p);
            fence_proxy_async();
            mbar_arrive(bar(BAR_KV_FULL + s));
            if (cached) {
                // staging slot s is consumed; thread 0 refills it with tile j + 2 once
                // every producer has arrived (a bounded wait, like all others)
                mbar_arrive(bar(BAR_STG_EMPTY + s));
                if (p == 0 && j + 2 < T && tile_of(j + 2) < n_cache_tiles &&
                    mbar_wait(bar(BAR_STG_EMPTY + s), (j >> 1) & 1, &abort_flag, err, 10))
                    stage_copy(j + 2);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int i = tid;                          // query row = TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const float sc = tau * kLog2e;
        const float jt = jensen == KV_JENSEN_TAYLOR2 ? tau * tau * (1.0f / 24.0f) * kLog2e : 0.5f * tau;
        // l_run sums the fp16-rounded P that the PV product consumes (so O / l_run
        // is a properly normalised average); l_ex sums the unrounded p for the lse.
        float m_ref = -INFINITY, l_run = 0.0f, l_ex = 0.0f;
        float x[kN];
        for (int j = 0; j < T; ++j) {
            const int s = j & 1;
            // the tile's metadata is ready: compute the Jensen terms while Q K^T runs
            const bool ok0 = mbar_wait(bar(BAR_KV_FULL + s), (j >> 1) & 1, &abort_flag, err, 4);
            if (!__all_sync(0xffffffffu, ok0)) break;
            const TileInfo info = reinterpret_cast<const TileInfo*>(sm + kInfoOff)[s];
            float dl[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (info.quantised && jensen != KV_JENSEN_OFF) {
                const float4* W4 = reinterpret_cast<const float4*>(sm + kWOff) + s * kD;   // [4][32] float4
#pragma unroll 2
                for (int ch = 0; ch < 16; ++ch) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sm + kQOff + sw_off(i, ch));
                    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                    float qf[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        qf[k] = __uint_as_float(k & 1 ? (qw[k >> 1] & 0xFFFF0000u) : (qw[k >> 1] << 16));
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float4 wa = W4[g * 32 + 2 * ch], wb = W4[g * 32 + 2 * ch + 1];
                        const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
                        if (jensen == KV_JENSEN_TAYLOR2) {
#pragma unroll
                            for (int k = 0; k < 8; ++k) dl[g] = fmaf(qf[k] * qf[k], w[k], dl[g]);
                        } else {
#pragma unroll
                            for (int k = 0; k < 8; ++k) dl[g] += log_sinhc(jt * qf[k] * w[k]);
                        }
                    }
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) dl[g] *= (jensen == KV_JENSEN_TAYLOR2 ? jt : kLog2e);
            }
            const bool ok1 = mbar_wait(bar(BAR_S_FULL + s), (j >> 1) & 1, &abort_flag, err, 5);
            if (!__all_sync(0xffffffffu, ok1)) break;
            fence_after();
#pragma unroll
            for (int g = 0; g < 4; ++g) tmem_ld32(tmem + lane_addr + s * kN + 32 * g, x + 32 * g);
            float mt = -INFINITY;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int nv = info.nvalid[g];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float v = k < nv ? fmaf(x[32 * g + k], sc, -dl[g]) : -INFINITY;
                    x[32 * g + k] = v;
                    mt = fmaxf(mt, v);
                }
            }
            const float m_new = fmaxf(m_ref, mt);
            const bool grow = m_new > m_ref + 8.0f;       // also true for the first finite max
            const bool ok2 = j == 0 || mbar_wait(bar(BAR_O_DONE), (j - 1) & 1, &abort_flag, err, 6);
            if (!__all_sync(0xffffffffu, ok2)) break;
            fence_after();
            // O is rescaled in TMEM when any row of the warp needs it; tcgen05.ld/st
            // are warp-collective, so the whole warp takes the branch (alpha = 1 for
            // rows whose running max did not move).
            const bool resc = grow && j > 0 && m_ref != -INFINITY;
            const float alpha = resc ? ex2(m_ref - m_new) : 1.0f;
            if (__any_sync(0xffffffffu, resc)) {
                float ob[32];
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    tmem_ld32(tmem + lane_addr + 256 + 32 * g, ob);
#pragma unroll
                    for (int k = 0; k < 32; ++k) ob[k] *= alpha;
                    tmem_st32(tmem + lane_addr + 256 + 32 * g, ob);
                }
            }
            l_run *= alpha;
            l_ex *= alpha;
            if (grow) m_ref = m_new;
            const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
            float psum = 0.0f, rsum = 0.0f;
            unsigned char* P = sm + kPOff;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                float pv[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    pv[k] = ex2(x[ch * 8 + k] - m_use);
                    psum += pv[k];
                }
                uint4 pk;
                pk.x = pack_f16(pv[0], pv[1]);
                pk.y = pack_f16(pv[2], pv[3]);
                pk.z = pack_f16(pv[4], pv[5]);
                pk.w = pack_f16(pv[6], pv[7]);
                const uint32_t pw[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pw[k]));
                    rsum += f.x + f.y;
                }
                *reinterpret_cast<uint4*>(P + sw_off(i, ch)) = pk;
            }
            l_run += rsum;
            l_ex += psum;
            fence_proxy_async();
            fence_before();
            mbar_arrive(bar(BAR_P_FULL));
        }
        // ---- epilogue
        const int qi = q0 + i;
        const long long orow = ((long long)b * Hq + hq) * n_q + qi;
        bool have = T > 0 && !abort_flag;
        if (have) have = mbar_wait(bar(BAR_O_DONE), (T - 1) & 1, &abort_flag, err, 7);
        have = __all_sync(0xffffffffu, have);
        fence_after();
        const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
        const long long rows = (long long)c.B * Hq * n_q;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            float ob[32];
            __syncwarp();
            if (have) {
                tmem_ld32(tmem + lane_addr + 256 + 32 * g, ob);
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
                if (lse) lse[orow] = (m_ref + log2f(l_ex)) * kLn2;
            } else {
                ws_ml[(long long)split * rows + orow] = make_float2(l_run > 0.0f ? m_ref * kLn2 : -INFINITY, l_run);
            }
        }
        __syncwarp();
    }
    fence_before();
    __syncthreads();
    if (warp == 8) {
        fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
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

}  // namespace

bool tc_supported(const kv_cache* cache, kv_dtype dt, int n_q, int Hq, const char** why) {
    const kv_layout& L = cache->layout;
    (void)Hq;
    if (dt != KV_BF16) { *why = "needs bf16 I/O"; return false; }
    if (L.d != kD) { *why = "needs head dim 128"; return false; }
    if (L.kind != KV_UNIFORM2 && L.kind != KV_UNIFORM4) { *why = "needs a UNIFORM2 or UNIFORM4 cache"; return false; }
    if (n_q < 16) { *why = "needs at least 16 queries"; return false; }
    return true;
}

int tc_auto_splits(const kv_cache* cache, int n_q, int n_cur, int Hq) {
    const kv_layout& L = cache->layout;
    const int seg = L.kind == KV_UNIFORM4 ? KV_SEG_INT4 : KV_SEG_INT2;
    const int tiles = (cache->n_blocks[seg] + 3) / 4 + (n_cur + kN - 1) / kN;
    const long long ctas = (long long)L.B * Hq * ((n_q + kM - 1) / kM);
    const int sms = num_sms();
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= 8; ++s) {
        if (s > 1 && tiles / s < 6) break;
        const double waves = (double)((ctas * s + sms - 1) / sms);
        const double cost = waves * ((double)tiles / s + 3.0);   // +3 tiles of pipeline fill per CTA
        if (cost < best_cost * 0.97) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

size_t tc_workspace(const kv_cache* cache, int n_q, int Hq, int n_splits) {
    size_t ws = 256;  // error word of the bounded waits
    if (n_splits > 1) {
        const long long rows = (long long)cache->layout.B * Hq * n_q;
        ws += (size_t)n_splits * rows * (kD * sizeof(float) + sizeof(float2));
    }
    return ws;
}

kv_status launch_attn_tc(const void* Q, const void* Kc, const void* Vc, int n_q, int n_cur, int Hq,
                         const kv_cache* cache, float tau, int jensen, int psac, int n_splits, void* out, int out_f32,
                         float* lse, void* ws, cudaStream_t st) {
    (void)psac;
    const DevCache c = make_dev_cache(cache);
    int* err = static_cast<int*>(ws);
    float* ws_o = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + 256);
    const long long rows = (long long)c.B * Hq * n_q;
    float2* ws_ml = reinterpret_cast<float2*>(ws_o + (n_splits > 1 ? (long long)n_splits * rows * kD : 0));
    const int n_qt = (n_q + kM - 1) / kM;
    dim3 grid(n_qt * n_splits, Hq, c.B);
    cudaMemsetAsync(err, 0, sizeof(int), st);
    static bool attr2 = false, attr4 = false;
    if (c.kind == KV_UNIFORM4) {
        if (!attr4) {
            cudaFuncSetAttribute(attn_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            attr4 = true;
        }
        attn_tc_kernel<4><<<grid, kThreads, kSmemBytes, st>>>(
            static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(Kc),
            static_cast<const __nv_bfloat16*>(Vc), n_q, n_cur, Hq, c, tau, jensen, n_splits, out, out_f32, lse, ws_o,
            ws_ml, err);
    } else {
        if (!attr2) {
            cudaFuncSetAttribute(attn_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            attr2 = true;
        }
        attn_tc_kernel<2><<<grid, kThreads, kSmemBytes, st>>>(
            static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(Kc),
            static_cast<const __nv_bfloat16*>(Vc), n_q, n_cur, Hq, c, tau, jensen, n_splits, out, out_f32, lse, ws_o,
            ws_ml, err);
    }
    kv_status s = check_launch("attn_tc_kernel");
    if (s != KV_OK) return s;
    if (getenv("BITKV_DEBUG_SYNC")) {
        int h_err = 0;
        cudaMemcpyAsync(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost, st);
        cudaStreamSynchronize(st);
        if (h_err) return set_error(KV_ERR_TIMEOUT, "attn_tc_kernel: bounded wait %d gave up", h_err);
    }
    if (n_splits == 1) return KV_OK;
    return launch_lse_merge(KV_BF16, ws_o, ws_ml, n_splits, rows, kD, out, out_f32, lse, st);
}

}  // namespace bitkv
