// sdpa_tc.cu -- tcgen05 tensor-core kernels of the materialised-probability
// SDPA forward (fp16 / bf16, head dim 64 or 128, positive scale): the
// two-pass kernel (one or two 128-row query tiles per CTA) and the fused
// single-sweep kernel for row blocks with at most two live 128-key tiles.
//
// What they compute: FlagOS-OP PR #10 "feat: add sdpa_math operator" -- the
// math backend's (out, attn_probs): P = softmax(scale*QK^T + mask), O = P V,
// with a fully masked row giving P = O = 0.  P is normalised exactly through
// the row log-sum-exp, the identity of the page's "P800 exact-P fast path"
// update (P = exp(scale*QK^T - LSE)), which the two-pass kernel evaluates in
// place:
//
//   sweep 1  S_j = Q K_j^T on the tensor cores (TMEM accumulator); running
//            row max / sum of exp2 in the softmax warps -> lse per row;
//   sweep 2  S_j again; p = exp2(S_j*scale*log2e - lse*log2e) written once
//            as dtype into a 128B-swizzled shared tile that is both the A
//            operand of O += P_j V_j (tensor cores) and the source of the TMA
//            stores of P.  Key tiles above a causal diagonal are never
//            computed; their P region is written with zeros.
//
// Two-pass kernel: one CTA owns one or two query tiles of one (batch, head);
// 12 warps:
//   warp 0       TMA producer (Q once; K tiles; then K/V tiles interleaved)
//   warp 1       TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2, 3   zero-fill of the P tiles above the causal diagonal
//   warps 4..11  two softmax warpgroups ("workers"), each with its own S
//                buffer in TMEM and P tile in shared memory
// Each softmax thread owns one query row (its TMEM lane).  With one query
// tile the workers alternate over its key tiles and merge their row
// statistics through shared memory after sweep 1; with two, worker s owns
// query tile s (see Work).  Each softmax warp stores its own 32 rows of every
// P tile with TMA as soon as it has written them.  After set-up the producer /
// MMA warpgroup hands registers to the softmax warpgroups.
//
// Every mbarrier wait is bounded: a wait that runs out records itself in the
// device status word and the CTA unwinds (freeing TMEM) instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace sdpa {

__device__ unsigned int g_status_word;

namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kWaitLimitCycles = 2000000000ll;  // ~1 s at GB300 clocks
constexpr int kThreads = 384;
// Register split after set-up: warpgroup 0 (producer / MMA / zero-fill warps)
// gives registers up, the two softmax warpgroups take them.  The launch must
// provide at least 128*kRegsLow + 256*kRegsHigh registers per CTA (checked on
// the host before the first launch; setmaxnreg.inc would otherwise wait forever).
constexpr uint32_t kRegsLow = 72, kRegsHigh = 208;

// The three outer tensor-map dimensions are stored in stride order; a packed
// code (2 bits per slot) says which logical dimension (1 = rows, 2 = head,
// 3 = batch) sits at tensor-map dim k+1, and pick() maps coordinates to it.
// Code 0 marks a broadcast dimension (stride 0 in the caller's view): the map
// holds it with extent 1 and every coordinate along it is 0.
__device__ __forceinline__ int pick(uint32_t sel, int rows, int head, int batch) {
    return sel == 1 ? rows : (sel == 2 ? head : (sel == 3 ? batch : 0));
}

struct TcParams {
    int Sq, Skv, Hq, group, n_qtiles, causal;
    int B, cl;  // batch; CTAs per cluster (one-sweep kernel)
    float c2;  // scale * log2(e), > 0
    const void* mask;
    int mask_kind, mask_dtype;
    long long sm0, sm1, sm2;
    void* o;
    long long so0, so1, so2;
    float* lse;
    void* p;  // P (the zero tiles above a causal diagonal are written with plain stores)
    long long sp0, sp1, sp2;
    uint32_t ord_q, ord_k, ord_v, ord_p, ord_o;
};

// Bounded mbarrier wait.  Returns false (after recording the first failure
// in the device status word and raising the CTA abort flag) if the phase does
// not complete within kWaitLimitCycles, or if another thread already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t role, uint32_t idx) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            const uint32_t blk = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
            atomicCAS(&g_status_word, 0u, (role << 24) | ((idx & 0xffu) << 16) | (blk & 0xffffu));
            return false;
        }
    }
    return true;
}

template <typename T> struct Pack;
template <> struct Pack<__half> {
    static __device__ __forceinline__ uint32_t two(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float load_bits(uint32_t bits) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    }
    static __device__ __forceinline__ float load(const void* p) { return __half2float(*(const __half*)p); }
};
template <> struct Pack<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t two(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float load_bits(uint32_t bits) {
        return __uint_as_float(bits << 16);
    }
    static __device__ __forceinline__ float load(const void* p) {
        return __bfloat162float(*(const __nv_bfloat16*)p);
    }
};

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
__device__ __forceinline__ uint16_t bits16(__half x) { return __half_as_ushort(x); }
__device__ __forceinline__ uint16_t bits16(__nv_bfloat16 x) { return __bfloat16_as_ushort(x); }

// Base-2 additive term of a user mask at (row, key): 0 / -inf for a bool
// mask, mask*log2(e) for an additive one.  Row and key must be in range.
template <typename T>
__device__ __forceinline__ float mask_term(const TcParams& p, int b, int h, int row, int key) {
    const long long off = b * p.sm0 + h * p.sm1 + row * p.sm2 + key;
    if (p.mask_kind == kMaskBool)
        return static_cast<const unsigned char*>(p.mask)[off] ? 0.f : -CUDART_INF_F;
    float m;
    if (p.mask_dtype == kF32) m = static_cast<const float*>(p.mask)[off];
    else m = Pack<T>::load(static_cast<const T*>(p.mask) + off);
    return m * kLog2e;
}

// ---------------------------------------------------------------- softmax tile helpers
// s[] holds one row of a 128-key score tile.  Without a user mask it holds the
// raw Q.K dot products (the base-2 scale is applied inside the exp2 FFMA,
// cexp = scale*log2e); with a user mask it is scaled and masked first
// (cexp = 1).  Masked entries are -inf either way.

template <typename T, bool kMasked, int NC = 128>
__device__ __forceinline__ void mask_tile(float (&s)[NC], const TcParams& prm, int b, int h, int row,
                                          bool row_ok, int kv0) {
    static_assert(NC % 4 == 0, "whole 32-bit mask words");
    if constexpr (kMasked) {
        const int n = row_ok ? min(NC, prm.Skv - kv0) : 0;  // keys of this row inside the tile
        const unsigned char* mrow = static_cast<const unsigned char*>(prm.mask) + b * prm.sm0 + h * prm.sm1 +
                                    (long long)row * prm.sm2 + kv0;
        if (prm.mask_kind == kMaskBool && n > 0 && (reinterpret_cast<uintptr_t>(mrow) & 3) == 0) {
            // bool mask: four keys per 32-bit load (the per-key byte loads of a
            // row-per-thread layout would each cost a separate memory request)
#pragma unroll
            for (int w = 0; w < NC / 4; ++w) {
                uint32_t m4 = 0;
                if (4 * w + 4 <= n) {
                    m4 = *reinterpret_cast<const uint32_t*>(mrow + 4 * w);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * w + e < n) m4 |= static_cast<uint32_t>(mrow[4 * w + e]) << (8 * e);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s[4 * w + e] = ((m4 >> (8 * e)) & 0xffu) ? fmaf(s[4 * w + e], prm.c2, 0.f) : -CUDART_INF_F;
            }
        } else {
#pragma unroll
            for (int x = 0; x < NC; ++x) {
                const float add = x < n ? mask_term<T>(prm, b, h, row, kv0 + x) : -CUDART_INF_F;
                s[x] = fmaf(s[x], prm.c2, add);
            }
        }
    }
    int lim = prm.Skv - 1 - kv0;  // last visible key offset in this tile
    if (prm.causal) lim = min(lim, row - kv0);
    if (!row_ok) lim = -1;
    if (lim < NC - 1) {
#pragma unroll
        for (int x = 0; x < NC; ++x) s[x] = (x > lim) ? -CUDART_INF_F : s[x];
    }
}

// Fold one tile into the running base-2 (max, sum of exp2) of the row.
__device__ __forceinline__ void tile_stats(const float (&s)[128], float cexp, float& m, float& l) {
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
    for (int x = 8; x < 128; ++x) mx[x & 7] = fmaxf(mx[x & 7], s[x]);
    const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                           fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cexp;
    const float mn = fmaxf(m, mt);
    if (mn != -CUDART_INF_F) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int x = 0; x < 128; ++x) acc[x & 7] += ex2(fmaf(s[x], cexp, -mn));
        l = l * ex2(m - mn) + (((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7])));
        m = mn;
    }
}

// p = exp2(s*cexp - lse2), packed to dtype pairs.  neg_lse is -lse2, or -inf
// for a fully masked row (every p becomes 0).
template <typename T>
__device__ __forceinline__ void tile_probs(const float (&s)[128], float cexp, float neg_lse, uint32_t (&hp)[64]) {
#pragma unroll
    for (int k = 0; k < 64; ++k)
        hp[k] = Pack<T>::two(ex2(fmaf(s[2 * k], cexp, neg_lse)), ex2(fmaf(s[2 * k + 1], cexp, neg_lse)));
}

// One row of a P tile into the 128B-swizzled shared layout (two 64-key chunks
// of 16 KB; 16-byte unit u of row t sits at unit u ^ (t % 8)).
__device__ __forceinline__ void store_p_row(const uint32_t (&hp)[64], uint32_t tile_base, int t) {
    const uint32_t rowaddr = tile_base + t * 128;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const uint32_t addr = rowaddr + (u / 8) * 16384 + (((u % 8) ^ (t % 8)) * 16);
        st_shared_v4(addr, hp[4 * u], hp[4 * u + 1], hp[4 * u + 2], hp[4 * u + 3]);
    }
}

// NCHUNK 64-column chunks of this thread's O row, from TMEM (fp32) into the
// 128B-swizzled staging tile (chunk c of row t at buf + c*16 KB + t*128,
// 16-byte unit u at u ^ (t % 8)), rounded to dtype; zeros for a dead row.
template <typename T, int NCHUNK>
__device__ __forceinline__ void stage_o_row(uint32_t taddr, uint32_t buf, int t, bool dead) {
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float ov[32];
            tmem_ld32(taddr + c * 64 + half * 32, ov);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = Pack<T>::two(dead ? 0.f : ov[u * 8 + 2 * e], dead ? 0.f : ov[u * 8 + 2 * e + 1]);
                const int unit = half * 4 + u;
                st_shared_v4(buf + c * 16384 + t * 128 + ((unit ^ (t % 8)) * 16), w[0], w[1], w[2], w[3]);
            }
        }
    }
}

// Per-warp P store: once a warp has written its 32 rows of a P tile into
// shared memory, its lane 0 stores them with two TMA boxes (64 keys x 32 rows
// each).  Before the warp rewrites that buffer, lane 0 waits until the bulk
// store has finished reading it.
__device__ __forceinline__ void warp_store_p(const CUtensorMap* tm, uint32_t ord, uint32_t tile_base, int w,
                                             int kv0, int r0, int h, int b) {
    const int row = r0 + 32 * w;
    for (int c = 0; c < 2; ++c)
        tma_store_4d(tm, tile_base + c * 16384 + w * 32 * 128, kv0 + 64 * c, pick(ord & 3, row, h, b),
                     pick((ord >> 2) & 3, row, h, b), pick((ord >> 4) & 3, row, h, b));
    bulk_commit();
}

// Per-warp O store: NCHUNK boxes of 64 columns x 32 rows from the staging
// tile, starting at output column col0.
template <int NCHUNK>
__device__ __forceinline__ void warp_store_o(const CUtensorMap* tm, uint32_t ord, uint32_t buf, int w, int col0,
                                             int r0, int h, int b) {
    const int row = r0 + 32 * w;
    for (int c = 0; c < NCHUNK; ++c)
        tma_store_4d(tm, buf + c * 16384 + w * 32 * 128, col0 + 64 * c, pick(ord & 3, row, h, b),
                     pick((ord >> 2) & 3, row, h, b), pick((ord >> 4) & 3, row, h, b));
    bulk_commit();
}

// Zero P[b, h, r0:r_end, z0:Skv] (the key tiles above a causal diagonal) with
// 16-byte stores: warp `w` of `nwarps` takes every nwarps-th row and its lanes
// cover consecutive 16-byte units of that row.  z0 is a multiple of 128 and
// rows are 16-byte aligned.
__device__ __forceinline__ void zero_p_region(const TcParams& prm, int b, int h, int r0, int r_end, int z0, int w,
                                              int nwarps, int lane) {
    if (z0 >= prm.Skv) return;
    const int n = prm.Skv - z0, nvec = n / 8;
    uint16_t* base = static_cast<uint16_t*>(prm.p) + b * prm.sp0 + h * prm.sp1 + z0;
    for (int r = r0 + w; r < r_end; r += nwarps) {
        uint16_t* row = base + (long long)r * prm.sp2;
        for (int k = lane; k < nvec; k += 32) *reinterpret_cast<uint4*>(row + 8 * k) = make_uint4(0u, 0u, 0u, 0u);
        if (lane < n - 8 * nvec) row[8 * nvec + lane] = 0;
    }
}

__device__ __forceinline__ void softmax_group_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int D, int QT>
struct TcCfg {
    static constexpr int kChunks = D / 64;               // 128-byte (64-element) column chunks
    static constexpr int kTileBytes = 128 * D * 2;        // one Q / K / V tile
    static constexpr int kPBytes = 128 * 128 * 2;         // one P tile (2 chunks)
    static constexpr int kBarBytes = 256;                 // mbarriers, TMEM slot, abort flag
    static constexpr int kFixed = QT * kTileBytes + 2 * kPBytes + kBarBytes + 1024;
    static constexpr int kMaxSmem = 227 * 1024;
    static constexpr int kStages = (kMaxSmem - kFixed) / kTileBytes > 8 ? 8 : (kMaxSmem - kFixed) / kTileBytes;
    static constexpr int kOffQ = 0;                        // QT query tiles
    static constexpr int kOffKV = kOffQ + QT * kTileBytes;
    static constexpr int kOffP = kOffKV + kStages * kTileBytes;  // one P tile per worker
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    // barrier indices
    static constexpr int bQ = 0;
    static constexpr int bKVF = 1;
    static constexpr int bKVE = bKVF + kStages;
    static constexpr int bSF = bKVE + kStages;   // [2] S buffer full  (MMA commit)
    static constexpr int bSE = bSF + 2;          // [2] S buffer empty (128 softmax threads)
    static constexpr int bPF = bSE + 2;          // [2] P buffer full  (128 softmax threads)
    static constexpr int bPV = bPF + 2;          // [2] P buffer consumed by P V (MMA commit)
    static constexpr int bO = bPV + 2;           // O complete (MMA commit)
    static constexpr int kBars = bO + 1;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemO = 256;  // O of stream s at kTmemO + s * D (QT == 2), else kTmemO
    static_assert(kBars * 8 + 16 <= kBarBytes, "barrier block");
    static_assert(kStages >= 2, "K/V ring too shallow");
    static_assert(kSmem <= kMaxSmem, "shared memory budget");
    static_assert(kTmemO + (QT == 2 ? 2 * D : D) <= kTmemCols, "TMEM budget");
};

// Which query tile(s) a CTA owns and how its score tiles are shared out.
// A unit is one 128x128 score tile (query tile s, key tile j); a CTA walks its
// units in key-tile order (both query tiles of key tile j before key tile
// j+1, so one K / V load feeds both) and hands each to one of its two softmax
// warpgroups ("workers"), which owns an S buffer and a P tile.
//   QT == 1: one 128-row query tile; unit j goes to worker j % 2, and the two
//            workers merge their row statistics after sweep 1.
//   QT == 2: two query tiles of one (batch, head); worker s owns query tile s
//            and all of its units.  (With a causal mask the tiles are paired
//            (i, n-1-i), which balances CTAs but not workers, so AUTO takes
//            this layout only without one.)
template <int QT>
struct Work {
    int q[2];      // query tile(s) (q[1] = -1: the CTA has one)
    int n[2];      // live key tiles of each query tile
    int n_kv;      // key tiles the CTA walks
    // is (query tile s, key tile j) a live unit?
    __device__ __forceinline__ bool has(int s, int j) const {
        if constexpr (QT == 2) return j < n[s];
        else return s == 0 && j < n_kv;
    }
};

__device__ __forceinline__ int live_tiles(const TcParams& p, int qt) {
    if (qt < 0) return 0;
    const int n_all = (p.Skv + 127) / 128;
    if (!p.causal) return n_all;
    const int r_last = min(qt * 128 + 127, p.Sq - 1);
    return min(r_last, p.Skv - 1) / 128 + 1;
}

template <int D, typename T, bool kMasked, int QT>
__global__ void __launch_bounds__(kThreads, 1)
tc_twopass_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
                  const __grid_constant__ CUtensorMap tm_o, const TcParams prm) {
    using C = TcCfg<D, QT>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int L = QT == 1 ? 2 : 1;  // sweep-2 lookahead of Q K^T over P V, in key tiles
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the shared-window offset (128B-swizzle atoms)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sKV = smem_u32(smem + C::kOffKV);
    const uint32_t sP = smem_u32(smem + C::kOffP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int hk = h / prm.group;
    Work<QT> wk;
    if constexpr (QT == 2) {
        wk.q[0] = blockIdx.z;
        wk.q[1] = prm.n_qtiles - 1 - (int)blockIdx.z;
        if (wk.q[1] <= wk.q[0]) wk.q[1] = -1;  // the middle tile of an odd count runs alone
        wk.n[0] = live_tiles(prm, wk.q[0]);
        wk.n[1] = live_tiles(prm, wk.q[1]);
        wk.n_kv = max(wk.n[0], wk.n[1]);
    } else {
        wk.q[0] = prm.n_qtiles - 1 - (int)blockIdx.z;  // heaviest causal tiles first
        wk.q[1] = -1;
        wk.n[0] = live_tiles(prm, wk.q[0]);
        wk.n[1] = 0;
        wk.n_kv = wk.n[0];
    }
    const int n_kv = wk.n_kv;

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kBars; ++i) mbar_init(bar(i), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::bSE + i), 128);
            mbar_init(bar(C::bPF + i), 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {  // producer / MMA / zero-fill warpgroup
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA producer
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const int nq = (QT == 2 && wk.q[1] >= 0) ? 2 : 1;
            mbar_arrive_expect_tx(bar(C::bQ), nq * C::kTileBytes);
            for (int s = 0; s < nq; ++s) {
                const int r0 = wk.q[s] * 128;
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(sQ + s * C::kTileBytes + c * 16384, &tm_q, bar(C::bQ), c * 64,
                                pick(prm.ord_q & 3, r0, h, b), pick((prm.ord_q >> 2) & 3, r0, h, b),
                                pick((prm.ord_q >> 4) & 3, r0, h, b));
            }
            int it = 0;
            auto load = [&](const CUtensorMap* tm, uint32_t ord, int kv0) {
                const int s = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1;
                wait_bar(bar(C::bKVE + s), ph ^ 1, abort_flag, 1, C::bKVE + s);
                mbar_arrive_expect_tx(bar(C::bKVF + s), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(sKV + s * C::kTileBytes + c * 16384, tm, bar(C::bKVF + s), c * 64,
                                pick(ord & 3, kv0, hk, b), pick((ord >> 2) & 3, kv0, hk, b),
                                pick((ord >> 4) & 3, kv0, hk, b));
                ++it;
            };
            // the MMA issuer consumes: K_0..K_{n-1} (sweep 1); then K_0..K_{L-1}
            // and, for each j, K_{j+L} (when it exists) followed by V_j (sweep 2)
            for (int j = 0; j < n_kv; ++j) load(&tm_k, prm.ord_k, j * 128);
            for (int j = 0; j < min(L, n_kv); ++j) load(&tm_k, prm.ord_k, j * 128);
            for (int j = 0; j < n_kv; ++j) {
                if (j + L < n_kv) load(&tm_k, prm.ord_k, (j + L) * 128);
                load(&tm_v, prm.ord_v, j * 128);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, kBF16, true);
            wait_bar(bar(C::bQ), 0, abort_flag, 2, C::bQ);
            int it = 0;
            int s_use0 = 0, s_use1 = 0, p_use0 = 0, p_use1 = 0;  // per worker (scalars: no local memory)
            bool o_init[2] = {false, false};                     // per query tile
            int uq = 0, up = 0;                          // units issued (Q K^T / P V) in this sweep
            // S = Q_s K_j^T for every live unit of key tile j, into its worker's S buffer
            auto qk = [&](int j) {
                const int st = it % C::kStages;
                wait_bar(bar(C::bKVF + st), (it / C::kStages) & 1, abort_flag, 2, C::bKVF + st);
#pragma unroll
                for (int s = 0; s < QT; ++s) {
                    if (!wk.has(s, j)) continue;
                    const int w = QT == 2 ? s : (uq & 1);  // QT == 2: stream s owns query tile s
                    ++uq;
                    const int use = w ? s_use1 : s_use0;
                    wait_bar(bar(C::bSE + w), (use & 1) ^ 1, abort_flag, 2, C::bSE + w);
                    tc_fence_after();
                    const uint32_t qbase = sQ + s * C::kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                        tc_mma_f16(tmem + w * 128, sw128_desc(qbase + off, 16, 1024),
                                   sw128_desc(sKV + st * C::kTileBytes + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(C::bSF + w));
                    if (w) ++s_use1;
                    else ++s_use0;
                }
                tc_commit(bar(C::bKVE + st));
                ++it;
            };
            // O_s += P V_j for every live unit of key tile j, from its worker's P tile
            auto pv = [&](int j) {
                const int st = it % C::kStages;
                wait_bar(bar(C::bKVF + st), (it / C::kStages) & 1, abort_flag, 2, C::bKVF + st);
#pragma unroll
                for (int s = 0; s < QT; ++s) {
                    if (!wk.has(s, j)) continue;
                    const int w = QT == 2 ? s : (up & 1);
                    ++up;
                    wait_bar(bar(C::bPF + w), (w ? p_use1 : p_use0) & 1, abort_flag, 2, C::bPF + w);
                    tc_fence_after();
                    const uint32_t od = tmem + C::kTmemO + s * D;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t a_off = (kk / 4) * 16384 + (kk % 4) * 32;  // P: K-major, 16 keys per step
                        const uint32_t b_off = kk * 2048;                         // V: N-major, 16 key rows per step
                        tc_mma_f16(od, sw128_desc(sP + w * C::kPBytes + a_off, 16, 1024),
                                   sw128_desc(sKV + st * C::kTileBytes + b_off, 16384, 1024), idesc_pv,
                                   (o_init[s] || kk > 0) ? 1u : 0u);
                    }
                    o_init[s] = true;
                    tc_commit(bar(C::bPV + w));
                    if (w) ++p_use1;
                    else ++p_use0;
                }
                tc_commit(bar(C::bKVE + st));
                ++it;
            };
            // sweep 1, then sweep 2 with Q K^T L key tiles ahead of P V, so that the
            // scores a worker needs next are computed while it writes P
            for (int j = 0; j < n_kv; ++j) qk(j);
            uq = 0;
            for (int j = 0; j < min(L, n_kv); ++j) qk(j);
            for (int j = 0; j < n_kv; ++j) {
                if (j + L < n_kv) qk(j + L);
                pv(j);
            }
            tc_commit(bar(C::bO));
        } else if (warp >= 2) {
            // ------------------------------------------------------------ causal zero tiles
            for (int s = 0; s < QT; ++s) {
                if (wk.q[s] < 0) continue;
                const int r0 = wk.q[s] * 128;
                zero_p_region(prm, b, h, r0, min(r0 + 128, prm.Sq), wk.n[s] * 128, warp - 2, 2, lane);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        setmaxnreg_inc<kRegsHigh>();
        if constexpr (QT == 2) {
            // two query tiles: stream s owns query tile s and all of its key tiles
            // (AUTO takes this layout only without a causal mask, where the two
            // streams hold the same number of tiles)
            const int sid = (warp - 4) >> 2;          // stream: S buffer, P buffer, barriers
            const int t = (threadIdx.x - 128) & 127;  // row within the tile == TMEM lane
            const int qt = wk.q[sid];
            if (qt >= 0) {
                const int r0 = qt * 128;
                const int row = r0 + t;
                const bool row_ok = row < prm.Sq;
                const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
                const uint32_t s_tmem = tmem + lane_base + sid * 128;
                const float cexp = kMasked ? 1.f : prm.c2;
                float s[128];
                int s_use = 0;

                auto load_s = [&](int role) {
                    wait_bar(bar(C::bSF + sid), s_use & 1, abort_flag, role, C::bSF + sid);
                    tc_fence_after();
                    tmem_ld128(s_tmem, s);
                    tc_fence_before();
                    mbar_arrive(bar(C::bSE + sid));
                    ++s_use;
                };

                // sweep 1: this stream's score tiles -> row max / sum of exp2
                float m = -CUDART_INF_F, l = 0.f;
                for (int j = 0; j < n_kv; ++j) {
                    if (!wk.has(sid, j)) continue;
                    load_s(4);
                    mask_tile<T, kMasked>(s, prm, b, h, row, row_ok, j * 128);
                    tile_stats(s, cexp, m, l);
                }
                const float lse2 = (m == -CUDART_INF_F) ? -CUDART_INF_F : m + log2f(l);
                const bool dead = lse2 == -CUDART_INF_F;
                const float neg_lse = dead ? -CUDART_INF_F : -lse2;  // a dead row adds -inf: every p is 0
                if (lane == 0) {
                    prefetch_tmap(&tm_p);
                    prefetch_tmap(&tm_o);
                }

                // sweep 2: exact P into this stream's swizzled shared tile, then TMA stores
                int p_use = 0;
                for (int j = 0; j < n_kv; ++j) {
                    if (!wk.has(sid, j)) continue;
                    load_s(5);
                    mask_tile<T, kMasked>(s, prm, b, h, row, row_ok, j * 128);
                    uint32_t hp[64];
                    tile_probs<T>(s, cexp, neg_lse, hp);
                    wait_bar(bar(C::bPV + sid), (p_use & 1) ^ 1, abort_flag, 5, C::bPV + sid);
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                    store_p_row(hp, sP + sid * C::kPBytes, t);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(C::bPF + sid));
                    __syncwarp();
                    if (lane == 0) warp_store_p(&tm_p, prm.ord_p, sP + sid * C::kPBytes, warp & 3, j * 128, r0, h, b);
                    ++p_use;
                }
                if (lane == 0) bulk_wait0();  // the P tile is read out before O reuses it
                __syncwarp();

                // epilogue: O rows (all D columns) from TMEM into this stream's (now
                // idle) P tile, then per-warp TMA stores
                wait_bar(bar(C::bO), 0, abort_flag, 6, C::bO);
                tc_fence_after();
                const uint32_t obuf = sP + sid * C::kPBytes;
                const uint32_t o_tmem = tmem + lane_base + C::kTmemO + sid * D;
                stage_o_row<T, D / 64>(o_tmem, obuf, t, dead);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) warp_store_o<D / 64>(&tm_o, prm.ord_o, obuf, warp & 3, 0, r0, h, b);
                if (lane == 0) bulk_wait0();
                if (prm.lse && row_ok)
                    prm.lse[((long long)b * prm.Hq + h) * prm.Sq + row] = dead ? lse2 : lse2 * kLn2;
            }
        } else {
            const int w = (warp - 4) >> 2;            // worker: S buffer, P tile, barriers
            const int t = (threadIdx.x - 128) & 127;  // row within a query tile == TMEM lane
            const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t s_tmem = tmem + lane_base + w * 128;
            const float cexp = kMasked ? 1.f : prm.c2;
            float s[128];
            int s_use = 0;

            auto load_s = [&](int role) {
                wait_bar(bar(C::bSF + w), s_use & 1, abort_flag, role, C::bSF + w);
                tc_fence_after();
                tmem_ld128(s_tmem, s);
                tc_fence_before();
                mbar_arrive(bar(C::bSE + w));
                ++s_use;
            };

            // sweep 1: this worker's units -> partial row max / sum of exp2 per query
            // tile.  The running pair of each (worker, query tile) lives in the
            // still idle P tiles, not in registers, so the unit loop carries no
            // per-tile state (and keeps one copy of its body).
            float* xs = reinterpret_cast<float*>(smem + C::kOffP);  // [worker][query tile][m, l][128]
    #pragma unroll
            for (int q = 0; q < QT; ++q) {
                xs[((w * QT + q) * 2 + 0) * 128 + t] = -CUDART_INF_F;
                xs[((w * QT + q) * 2 + 1) * 128 + t] = 0.f;
            }
            int u = 0;
            for (int j = 0; j < n_kv; ++j) {
    #pragma unroll 1
                for (int q = 0; q < QT; ++q) {
                    if (!wk.has(q, j)) continue;
                    if ((u++ & 1) != w) continue;
                    const int row = (q ? wk.q[1] : wk.q[0]) * 128 + t;
                    load_s(4);
                    mask_tile<T, kMasked>(s, prm, b, h, row, row < prm.Sq, j * 128);
                    float* st = xs + ((w * QT + q) * 2) * 128 + t;
                    float mq = st[0], lq = st[128];
                    tile_stats(s, cexp, mq, lq);
                    st[0] = mq;
                    st[128] = lq;
                }
            }
            // merge the two workers' statistics: both combine the same values in the
            // same order, so they hold bit-identical lse per row
            softmax_group_sync();
            float lse2_0 = -CUDART_INF_F, lse2_1 = -CUDART_INF_F;
    #pragma unroll
            for (int q = 0; q < QT; ++q) {
                const float a0 = xs[((0 * QT + q) * 2 + 0) * 128 + t], b0 = xs[((0 * QT + q) * 2 + 1) * 128 + t];
                const float a1 = xs[((1 * QT + q) * 2 + 0) * 128 + t], b1 = xs[((1 * QT + q) * 2 + 1) * 128 + t];
                const float mm = fmaxf(a0, a1);
                const float v = (mm == -CUDART_INF_F) ? -CUDART_INF_F : mm + log2f(b0 * ex2(a0 - mm) + b1 * ex2(a1 - mm));
                if (q) lse2_1 = v;
                else lse2_0 = v;
            }
            softmax_group_sync();  // both read the exchange before any P tile is written
            if (lane == 0) {
                prefetch_tmap(&tm_p);
                prefetch_tmap(&tm_o);
            }

            // sweep 2: exact P of this worker's units into its swizzled P tile, then TMA stores
            int p_use = 0;
            u = 0;
            const float neg0 = lse2_0 == -CUDART_INF_F ? -CUDART_INF_F : -lse2_0;  // a dead row adds -inf: p = 0
            const float neg1 = lse2_1 == -CUDART_INF_F ? -CUDART_INF_F : -lse2_1;
            for (int j = 0; j < n_kv; ++j) {
    #pragma unroll 1
                for (int q = 0; q < QT; ++q) {
                    if (!wk.has(q, j)) continue;
                    if ((u++ & 1) != w) continue;
                    const int r0 = (q ? wk.q[1] : wk.q[0]) * 128, row = r0 + t;
                    load_s(5);
                    mask_tile<T, kMasked>(s, prm, b, h, row, row < prm.Sq, j * 128);
                    uint32_t hp[64];
                    tile_probs<T>(s, cexp, q ? neg1 : neg0, hp);
                    wait_bar(bar(C::bPV + w), (p_use & 1) ^ 1, abort_flag, 5, C::bPV + w);
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                    store_p_row(hp, sP + w * C::kPBytes, t);
                    fence_proxy_async_smem();
                    mbar_arrive(bar(C::bPF + w));
                    __syncwarp();
                    if (lane == 0) warp_store_p(&tm_p, prm.ord_p, sP + w * C::kPBytes, warp & 3, j * 128, r0, h, b);
                    ++p_use;
                }
            }
            if (lane == 0) bulk_wait0();  // the P tile is read out before O reuses it
            __syncwarp();

            // epilogue: O rows from TMEM into this worker's (now idle) P tile, then
            // per-warp TMA stores.  QT == 2: worker w writes query tile w (all D
            // columns); QT == 1: worker w takes the 64-column chunk w (D = 128), or
            // worker 0 all 64 columns (D = 64).
            wait_bar(bar(C::bO), 0, abort_flag, 6, C::bO);
            tc_fence_after();
            const uint32_t obuf = sP + w * C::kPBytes;
            const int oq = QT == 2 ? w : 0;  // query tile whose O this worker writes
            if (wk.q[oq] >= 0) {
                const int r0 = wk.q[oq] * 128, row = r0 + t;
                const bool row_ok = row < prm.Sq;
                const float lse_o = oq ? lse2_1 : lse2_0;
                const bool dead = lse_o == -CUDART_INF_F;
                const uint32_t o_tmem = tmem + lane_base + C::kTmemO + oq * D;
                if constexpr (QT == 2) {
                    stage_o_row<T, D / 64>(o_tmem, obuf, t, dead);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) warp_store_o<D / 64>(&tm_o, prm.ord_o, obuf, warp & 3, 0, r0, h, b);
                } else if (D == 128 || w == 0) {
                    const int c0 = D == 128 ? w : 0;
                    stage_o_row<T, 1>(o_tmem + 64 * c0, obuf, t, dead);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) warp_store_o<1>(&tm_o, prm.ord_o, obuf, warp & 3, 64 * c0, r0, h, b);
                }
                if (lane == 0) bulk_wait0();
                if ((QT == 2 || w == 0) && prm.lse && row_ok)
                    prm.lse[((long long)b * prm.Hq + h) * prm.Sq + row] = dead ? lse_o : lse_o * kLn2;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (*abort_flag) {
            // give in-flight TMA / tcgen05 work time to land before freeing TMEM
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        }
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- two-pass kernel, 256-key score tiles
// One 128-row query tile per CTA (causal calls, and grids the paired layout
// cannot fill).  Q K^T runs over pairs of key tiles as 128 x 256 x 16 MMAs
// with Q in TMEM as the A operand: on GB300 such an instruction takes ~137
// cycles against ~107 for a 128 x 128 x 16 one with both operands in shared
// memory, so the score products of both sweeps cost about 0.64x of the
// 128-key form.  P V stays 128 x D x 16 with P from the worker's shared tile.
//
// TMEM (512 columns): S of a key-tile pair in [0, 256) (worker w reads
// [128 w, 128 w + 128)), O in [256, 256 + D), Q in [384, 384 + D / 2) as
// packed element pairs.  Shared memory: a ring of pair slots (two K tiles laid
// out as one 256-row operand, chunk c of tile t at c * 32 KB + t * 16 KB; or
// two V tiles one after the other) and one P tile per worker; P tile 0 holds
// the Q tile until worker 0 has copied it into TMEM.
//   warp 0       TMA producer: Q, K pairs (sweep 1), then K pairs and V pairs
//   warp 1       TMEM allocator + MMA issuer
//   warps 2, 3   zero-fill of P above the causal diagonal
//   warps 4..11  two softmax workers; worker w takes key tile 2 p + w of pair p
template <int D>
struct WideCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = 128 * D * 2;      // one 128-row Q / K / V tile
    static constexpr int kSlot = 2 * kTile;        // a pair of K or V tiles
    static constexpr int kPBytes = 128 * 128 * 2;  // one P tile
    static constexpr int kBarBytes = 256;
    static constexpr int kMaxSmem = 227 * 1024;
    static constexpr int kFree = kMaxSmem - 2 * kPBytes - kBarBytes - 1024;
    static constexpr int kSlots = kFree / kSlot > 6 ? 6 : kFree / kSlot;
    static constexpr int kOffRing = 0;
    static constexpr int kOffP = kSlots * kSlot;
    static constexpr int kOffBar = kOffP + 2 * kPBytes;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack
    static constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;
    static constexpr int bQ = 0;             // Q tile landed in P tile 0 (TMA)
    static constexpr int bQT = 1;            // Q in TMEM (128 arrivals)
    static constexpr int bF = 2;             // [kSlots] slot full (TMA)
    static constexpr int bE = bF + kSlots;   // [kSlots] slot consumed (MMA commit)
    static constexpr int bSF = bE + kSlots;  // S full (MMA commit)
    static constexpr int bSE = bSF + 1;      // S read out by both workers (256 arrivals)
    static constexpr int bPF = bSE + 1;      // [2] P tile full (128 arrivals)
    static constexpr int bPV = bPF + 2;      // [2] P tile consumed by P V (MMA commit)
    static constexpr int bO = bPV + 2;       // O complete (MMA commit)
    static constexpr int kBars = bO + 1;
    static_assert(kBars * 8 + 16 <= kBarBytes, "barrier block");
    static_assert(kSlots >= 2, "ring too shallow");
    static_assert(kSmem <= kMaxSmem, "shared memory budget");
    static_assert(kColO + D <= kColQ && kColQ + D / 2 <= 512, "TMEM budget");
};

template <int D, typename T, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
tc_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
               const __grid_constant__ CUtensorMap tm_o, const TcParams prm) {
    using C = WideCfg<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sRing = smem_u32(smem + C::kOffRing);
    const uint32_t sP = smem_u32(smem + C::kOffP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int hk = h / prm.group;
    const int qt = prm.n_qtiles - 1 - (int)blockIdx.z;  // heaviest causal tiles first
    const int r0 = qt * 128;
    const int n = live_tiles(prm, qt);                  // live key tiles
    const int np = (n + 1) / 2;                         // key-tile pairs

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kBars; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(C::bQT), 128);
        mbar_init(bar(C::bSE), 256);
        mbar_init(bar(C::bPF), 128);
        mbar_init(bar(C::bPF + 1), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {  // producer / MMA / zero-fill warpgroup
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA producer
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(bar(C::bQ), C::kTile);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(sP + c * 16384, &tm_q, bar(C::bQ), c * 64, pick(prm.ord_q & 3, r0, h, b),
                            pick((prm.ord_q >> 2) & 3, r0, h, b), pick((prm.ord_q >> 4) & 3, r0, h, b));
            int it = 0;
            auto load_pair = [&](const CUtensorMap* tm, uint32_t ord, int p, bool is_k) {
                const int s = it % C::kSlots;
                wait_bar(bar(C::bE + s), ((it / C::kSlots) & 1) ^ 1, abort_flag, 1, C::bE + s);
                const int nt = min(2, n - 2 * p);
                mbar_arrive_expect_tx(bar(C::bF + s), nt * C::kTile);
                for (int t = 0; t < nt; ++t) {
                    const int kv0 = (2 * p + t) * 128;
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(sRing + s * C::kSlot + (is_k ? c * 32768 + t * 16384 : t * C::kTile + c * 16384),
                                    tm, bar(C::bF + s), c * 64, pick(ord & 3, kv0, hk, b),
                                    pick((ord >> 2) & 3, kv0, hk, b), pick((ord >> 4) & 3, kv0, hk, b));
                }
                ++it;
            };
            // the MMA issuer consumes: K pairs 0..np-1 (sweep 1); then K pair 0 and,
            // for each pair p, K pair p+1 (when it exists) followed by V pair p
            for (int p = 0; p < np; ++p) load_pair(&tm_k, prm.ord_k, p, true);
            load_pair(&tm_k, prm.ord_k, 0, true);
            for (int p = 0; p < np; ++p) {
                if (p + 1 < np) load_pair(&tm_k, prm.ord_k, p + 1, true);
                load_pair(&tm_v, prm.ord_v, p, false);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_qk2 = idesc_f16(128, 256, kBF16, false);
            constexpr uint32_t idesc_qk1 = idesc_f16(128, 128, kBF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, kBF16, true);
            // descriptor bases: a slot, tile or K step adds its byte offset / 16
            // to the start-address field (addresses stay below 2^18 bytes)
            const uint64_t kdesc0 = sw128_desc(sRing, 16, 1024);
            const uint64_t vdesc0 = sw128_desc(sRing, 16384, 1024);
            const uint64_t pdesc0 = sw128_desc(sP, 16, 1024);
            wait_bar(bar(C::bQT), 0, abort_flag, 2, C::bQT);
            tc_fence_after();
            int it = 0, s_use = 0, pu0 = 0, pu1 = 0;
            bool o_init = false;
            // S = Q [K_2p | K_2p+1]^T (N = 256, or 128 for a lone last tile)
            auto qk = [&](int p) {
                const int s = it % C::kSlots;
                wait_bar(bar(C::bF + s), (it / C::kSlots) & 1, abort_flag, 2, C::bF + s);
                wait_bar(bar(C::bSE), (s_use & 1) ^ 1, abort_flag, 2, C::bSE);
                tc_fence_after();
                const uint64_t kd = kdesc0 + static_cast<uint64_t>((s * C::kSlot) >> 4);
                const uint32_t idesc = (2 * p + 1 < n) ? idesc_qk2 : idesc_qk1;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_f16_ts(tmem + C::kColS, tmem + C::kColQ + kk * 8,
                                  kd + static_cast<uint64_t>(((kk / 4) * 32768 + (kk % 4) * 32) >> 4), idesc,
                                  kk > 0 ? 1u : 0u);
                tc_commit(bar(C::bSF));
                tc_commit(bar(C::bE + s));
                ++it;
                ++s_use;
            };
            // O += P_t V_t for the tiles of pair p, P from worker t's tile
            auto pv = [&](int p) {
                const int s = it % C::kSlots;
                wait_bar(bar(C::bF + s), (it / C::kSlots) & 1, abort_flag, 2, C::bF + s);
                const int nt = min(2, n - 2 * p);
                for (int t = 0; t < nt; ++t) {
                    wait_bar(bar(C::bPF + t), (t ? pu1 : pu0) & 1, abort_flag, 2, C::bPF + t);
                    tc_fence_after();
                    const uint64_t vd = vdesc0 + static_cast<uint64_t>((s * C::kSlot + t * C::kTile) >> 4);
                    const uint64_t pd = pdesc0 + static_cast<uint64_t>((t * C::kPBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_f16(tmem + C::kColO, pd + static_cast<uint64_t>(((kk / 4) * 16384 + (kk % 4) * 32) >> 4),
                                   vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (o_init || kk > 0) ? 1u : 0u);
                    o_init = true;
                    tc_commit(bar(C::bPV + t));
                    if (t) ++pu1;
                    else ++pu0;
                }
                tc_commit(bar(C::bE + s));
                ++it;
            };
            // sweep 1, then sweep 2 with the next pair's Q K^T ahead of this pair's P V
            for (int p = 0; p < np; ++p) qk(p);
            qk(0);
            for (int p = 0; p < np; ++p) {
                if (p + 1 < np) qk(p + 1);
                pv(p);
            }
            tc_commit(bar(C::bO));
        } else if (warp >= 2) {
            // ------------------------------------------------------------ causal zero tiles
            zero_p_region(prm, b, h, r0, min(r0 + 128, prm.Sq), n * 128, warp - 2, 2, lane);
        }
    } else {
        // ------------------------------------------------------------ softmax workers
        setmaxnreg_inc<kRegsHigh>();
        const int w = (warp - 4) >> 2;
        const int t = (threadIdx.x - 128) & 127;  // row within the tile == TMEM lane
        const int row = r0 + t;
        const bool row_ok = row < prm.Sq;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_tmem = tmem + lane_base + C::kColS + w * 128;
        const float cexp = kMasked ? 1.f : prm.c2;

        // Q into TMEM (worker 0): row t of the swizzled tile in P tile 0, as
        // packed element pairs in columns [kColQ, kColQ + D / 2) of lane t
        if (w == 0) {
            wait_bar(bar(C::bQ), 0, abort_flag, 3, C::bQ);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                uint32_t qr[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 v4 = ld_shared_v4(sP + c * 16384 + t * 128 + ((u ^ (t % 8)) * 16));
                    qr[4 * u] = v4.x;
                    qr[4 * u + 1] = v4.y;
                    qr[4 * u + 2] = v4.z;
                    qr[4 * u + 3] = v4.w;
                }
                tmem_st32(tmem + lane_base + C::kColQ + c * 32, qr);
            }
            tc_fence_before();
            mbar_arrive(bar(C::bQT));
        }

        float s[128];
        int s_use = 0;
        // every pair's S: both workers wait for it and release it, in step
        auto load_s = [&](bool has, int role) {
            wait_bar(bar(C::bSF), s_use & 1, abort_flag, role, C::bSF);
            tc_fence_after();
            if (has) tmem_ld128(s_tmem, s);
            tc_fence_before();
            mbar_arrive(bar(C::bSE));
            ++s_use;
        };

        // sweep 1: this worker's tiles -> partial row max / sum of exp2
        float m = -CUDART_INF_F, l = 0.f;
        for (int p = 0; p < np; ++p) {
            const int j = 2 * p + w;
            const bool has = j < n;
            load_s(has, 4);
            if (has) {
                mask_tile<T, kMasked>(s, prm, b, h, row, row_ok, j * 128);
                tile_stats(s, cexp, m, l);
            }
        }
        // merge the two workers' statistics through P tile 1 (idle until
        // sweep 2): both combine the same values in the same order, so they
        // hold bit-identical lse per row
        float* xs = reinterpret_cast<float*>(smem + C::kOffP + C::kPBytes);  // [worker][m, l][128]
        xs[(w * 2 + 0) * 128 + t] = m;
        xs[(w * 2 + 1) * 128 + t] = l;
        softmax_group_sync();
        float lse2;
        {
            const float a0 = xs[t], b0 = xs[128 + t], a1 = xs[256 + t], b1 = xs[384 + t];
            const float mm = fmaxf(a0, a1);
            lse2 = (mm == -CUDART_INF_F) ? -CUDART_INF_F : mm + log2f(b0 * ex2(a0 - mm) + b1 * ex2(a1 - mm));
        }
        softmax_group_sync();  // both read the exchange before any P tile is written
        if (lane == 0) {
            prefetch_tmap(&tm_p);
            prefetch_tmap(&tm_o);
        }
        const bool dead = lse2 == -CUDART_INF_F;
        const float neg = dead ? -CUDART_INF_F : -lse2;  // a dead row adds -inf: every p is 0

        // sweep 2: exact P of this worker's tiles into its swizzled P tile, then TMA stores
        int p_use = 0;
        for (int p = 0; p < np; ++p) {
            const int j = 2 * p + w;
            const bool has = j < n;
            load_s(has, 5);
            if (!has) continue;
            mask_tile<T, kMasked>(s, prm, b, h, row, row_ok, j * 128);
            uint32_t hp[64];
            tile_probs<T>(s, cexp, neg, hp);
            wait_bar(bar(C::bPV + w), (p_use & 1) ^ 1, abort_flag, 5, C::bPV + w);
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
            store_p_row(hp, sP + w * C::kPBytes, t);
            fence_proxy_async_smem();
            mbar_arrive(bar(C::bPF + w));
            __syncwarp();
            if (lane == 0) warp_store_p(&tm_p, prm.ord_p, sP + w * C::kPBytes, warp & 3, j * 128, r0, h, b);
            ++p_use;
        }
        if (lane == 0) bulk_wait0();  // the P tile is read out before O reuses it
        __syncwarp();

        // epilogue: worker w stages and stores the 64-column chunk w of O
        // (D = 128), or worker 0 all of it (D = 64), through its idle P tile
        wait_bar(bar(C::bO), 0, abort_flag, 6, C::bO);
        tc_fence_after();
        if (D == 128 || w == 0) {
            const int c0 = D == 128 ? w : 0;
            const uint32_t obuf = sP + w * C::kPBytes;
            stage_o_row<T, 1>(tmem + lane_base + C::kColO + 64 * c0, obuf, t, dead);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) warp_store_o<1>(&tm_o, prm.ord_o, obuf, warp & 3, 64 * c0, r0, h, b);
            if (lane == 0) bulk_wait0();
        }
        if (w == 0 && prm.lse && row_ok)
            prm.lse[((long long)b * prm.Hq + h) * prm.Sq + row] = dead ? lse2 : lse2 * kLn2;
    }

    // ------------------------------------------------------------ teardown
    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (*abort_flag) {
            // give in-flight TMA / tcgen05 work time to land before freeing TMEM
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        }
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- one-sweep cluster kernel
// The whole forward in one Q K^T sweep.  The live key tiles of a 128-row
// query block are dealt round-robin over a cluster of C CTAs (tile j to CTA
// j % C, at most kMaxOwn tiles each), and every CTA keeps the exponentials of
// its tiles in TMEM instead of recomputing the scores:
//   A  S_j = Q K_j^T (tcgen05, TMEM); per row and per 64-key half tile the max
//      m_j, e = exp2(s - m_j) rounded to fp16 and kept in TMEM, and the row's
//      running (max, sum of exp2);
//   B  every CTA sends its rows' (max, sum) into each cluster CTA's shared
//      memory (st.async, completing on that CTA's mbarrier): every CTA then
//      holds the exact row LSE of the whole key range;
//   C  P = e * exp2(m_j - lse) in the output dtype, written back over e in TMEM
//      (the A operand of O_part += P V_j) and, per warp, into a 128B-swizzled
//      32 x 64 shared box that a TMA store copies to P;
//   D  every CTA sends the partial-O rows CTA c owns ([ceil(128 c / C),
//      ceil(128 (c + 1) / C))) from registers into c's shared memory
//      (st.async); c adds them to its own partial rows and stores O.
// P is normalised by the final LSE, as in the two-sweep form; the one extra
// rounding is that of e to fp16 (relative 2^-12 on values in (0, 1], so at
// most ~2.5e-4 absolute on P), inside the half-ulp of an f16 / bf16 P.
// K and V are read once per query block, Q K^T runs once and exp2 runs once
// per score.  Clusters are persistent over query blocks (heaviest causal
// blocks first, snake order over clusters).  All cross-CTA traffic is
// st.async into the receiver's shared memory, completing on the receiver's
// own mbarriers; the statistics of block k reach a CTA only after it has
// finished block k - 1, which orders every reuse of its receive slots.
//
// Shared memory: a ring of K / V tile slots, the Q tile (refilled for the
// next block once the last Q K^T has read it), one 32 x 64 P box per worker
// warp, the receive area (the peers' partial-O rows, then their statistics
// in its last C KB), the warpgroup merge area, barriers.  TMEM: S in
// [0, 128), e / P of own tile i in [128 + 64 i, 192 + 64 i) as packed 16-bit
// pairs (warpgroup g: 32 columns at + 32 g), O in [384, 384 + D).
//   warp 0       TMA producer: per block Q, then the CTA's K tiles, then its V tiles
//   warp 1       TMEM allocator + MMA issuer
//   warps 2, 3   zero-fill of this CTA's rows of P above the causal diagonal
//   warps 4..11  two softmax warpgroups; warpgroup g takes keys [64 g, 64 g + 64)
//                of every tile
template <int D>
struct OneCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = 128 * D * 2;      // one 128-row Q / K / V tile
    static constexpr int kMaxOwn = 4;              // key tiles a CTA keeps per query block
    static constexpr int kBoxBytes = 32 * 128;     // one warp's 32-row x 64-key P box
    static constexpr int kRecvBytes = 64 * 1024;   // partial-O rows of the peers + their statistics
    static constexpr int kMergeBytes = 1024;       // warpgroup 1's (max, sum) per row
    static constexpr int kBarBytes = 256;
    static constexpr int kMaxSmem = 227 * 1024;
    static constexpr int kFixed = kTile + 8 * kBoxBytes + kRecvBytes + kMergeBytes + kBarBytes + 1024;
    static constexpr int kSlots = (kMaxSmem - kFixed) / kTile > 6 ? 6 : (kMaxSmem - kFixed) / kTile;
    static constexpr int kOffRing = 0;
    static constexpr int kOffQ = kOffRing + kSlots * kTile;
    static constexpr int kOffBox = kOffQ + kTile;
    static constexpr int kOffRecv = kOffBox + 8 * kBoxBytes;
    static constexpr int kOffMerge = kOffRecv + kRecvBytes;
    static constexpr int kOffBar = kOffMerge + kMergeBytes;
    static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + alignment slack
    static constexpr uint32_t kColS = 0, kColE = 128, kColO = 384;
    static constexpr int bQF = 0;               // Q tile landed (TMA)
    static constexpr int bQE = 1;               // Q tile read by the block's last Q K^T (MMA commit)
    static constexpr int bF = 2;                // [kSlots] ring slot full (TMA)
    static constexpr int bE = bF + kSlots;      // [kSlots] ring slot consumed (MMA commit)
    static constexpr int bSF = bE + kSlots;     // S full (MMA commit)
    static constexpr int bSE = bSF + 1;         // S read out (256 worker arrivals)
    static constexpr int bPF = bSE + 1;         // [kMaxOwn] P of own tile i in TMEM (256 worker arrivals)
    static constexpr int bO = bPF + kMaxOwn;    // partial O complete (MMA commit)
    static constexpr int bOE = bO + 1;          // partial O read out of TMEM (one worker arrival)
    static constexpr int bST = bOE + 1;         // every cluster CTA's statistics landed (1 arrival + bytes)
    static constexpr int bRecv = bST + 1;       // the peers' partial-O rows landed (1 arrival + bytes)
    static constexpr int kBars = bRecv + 1;
    static_assert(kBars * 8 + 16 <= kBarBytes, "barrier block");
    static_assert(kSlots >= 3, "ring too shallow");
    // (C - 1) slots of ceil(128 / C) rows (at most 114 rows, C = 7) + C KB of
    // statistics, for every C <= 8
    static_assert(114 * D * 4 + 7 * 1024 <= kRecvBytes && 112 * D * 4 + 8 * 1024 <= kRecvBytes, "receive area");
    static_assert(kSmem <= kMaxSmem, "shared memory budget");
    static_assert(kColO + D <= 512 && kColE + 64 * kMaxOwn <= kColO, "TMEM budget");
};
constexpr int kOneMaxCluster = 8;  // portable cluster size: up to 32 live key tiles per query block

struct OneItem {
    int b, h, qt, n;  // batch, head, query tile, live key tiles
};

// Query blocks in decreasing causal weight: rank r -> query tile
// n_qtiles - 1 - r / (B * Hq), then (b, h).
__device__ __forceinline__ OneItem one_item(const TcParams& prm, int r) {
    const int bh = prm.B * prm.Hq;
    OneItem I;
    I.qt = prm.n_qtiles - 1 - r / bh;
    const int x = r % bh;
    I.b = x / prm.Hq;
    I.h = x % prm.Hq;
    I.n = live_tiles(prm, I.qt);
    return I;
}

// The k-th query block of cluster c among G clusters (snake order).
__device__ __forceinline__ int one_rank(int k, int c, int G) { return k * G + ((k & 1) ? G - 1 - c : c); }

// Bounded wait whose phase may be completed from a peer CTA (acquire at
// cluster scope).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 uint32_t role, uint32_t idx) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            atomicCAS(&g_status_word, 0u, (role << 24) | ((idx & 0xffu) << 16) | (blockIdx.x & 0xffffu));
            return false;
        }
    }
    return true;
}

template <int D, typename T, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
tc_onesweep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
                   const TcParams prm) {
    using C = OneCfg<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sRing = smem_u32(smem + C::kOffRing);
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sBox = smem_u32(smem + C::kOffBox);
    const uint32_t sRecv = smem_u32(smem + C::kOffRecv);
    float* mgM = reinterpret_cast<float*>(smem + C::kOffMerge);
    float* mgL = mgM + 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int CL = prm.cl;
    const uint32_t rank = cluster_ctarank();
    const int cl = (int)blockIdx.x / CL, G = (int)gridDim.x / CL;
    const int n_items = prm.B * prm.Hq * prm.n_qtiles;
    // key tiles of query block I this CTA owns: rank, rank + C, ...
    auto n_own_of = [&](const OneItem& I) { return I.n > (int)rank ? (I.n - (int)rank + CL - 1) / CL : 0; };
    // first O row of the slice CTA c reduces (row t belongs to CTA t * C / 128)
    auto row_begin = [&](int c) { return (c * 128 + CL - 1) / CL; };
    // the peers' statistics, float2 [C][128], in the last C KB of the receive area
    const uint32_t sStat = sRecv + C::kRecvBytes - CL * 1024;

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kBars; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(C::bSE), 256);
        for (int i = 0; i < C::kMaxOwn; ++i) mbar_init(bar(C::bPF + i), 256);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_barrier();  // barriers initialised in every CTA before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        setmaxnreg_dec<kRegsLow>();
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA producer
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int it = 0, q_use = 0;
            auto load_tile = [&](uint32_t dst, const CUtensorMap* tm, uint32_t full, uint32_t ord, int row0, int head,
                                 int b) {
                mbar_arrive_expect_tx(full, C::kTile);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(dst + c * 16384, tm, full, c * 64, pick(ord & 3, row0, head, b),
                                pick((ord >> 2) & 3, row0, head, b), pick((ord >> 4) & 3, row0, head, b));
            };
            auto load = [&](const CUtensorMap* tm, uint32_t ord, int row0, int head, int b) {
                const int s = it % C::kSlots;
                wait_bar(bar(C::bE + s), ((it / C::kSlots) & 1) ^ 1, abort_flag, 1, C::bE + s);
                load_tile(sRing + s * C::kTile, tm, bar(C::bF + s), ord, row0, head, b);
                ++it;
            };
            for (int k = 0;; ++k) {
                const int r = one_rank(k, cl, G);
                if (r >= n_items) break;
                const OneItem I = one_item(prm, r);
                const int no = n_own_of(I), hk = I.h / prm.group;
                if (no == 0) continue;
                wait_bar(bar(C::bQE), (q_use & 1) ^ 1, abort_flag, 1, C::bQE);
                load_tile(sQ, &tm_q, bar(C::bQF), prm.ord_q, I.qt * 128, I.h, I.b);
                ++q_use;
                for (int i = 0; i < no; ++i) load(&tm_k, prm.ord_k, ((int)rank + CL * i) * 128, hk, I.b);
                for (int i = 0; i < no; ++i) load(&tm_v, prm.ord_v, ((int)rank + CL * i) * 128, hk, I.b);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBF16, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, D, kBF16, true);
            const uint64_t rdesc0 = sw128_desc(sRing, 16, 1024);     // K: K-major
            const uint64_t qd = sw128_desc(sQ, 16, 1024);            // Q: K-major
            const uint64_t vdesc0 = sw128_desc(sRing, 16384, 1024);  // V: N-major, 64-column chunks 16 KB apart
            int it = 0, s_use = 0, q_use = 0;
            uint32_t pf_phase = 0;
            for (int k = 0;; ++k) {
                const int r = one_rank(k, cl, G);
                if (r >= n_items) break;
                const OneItem I = one_item(prm, r);
                const int no = n_own_of(I);
                if (no > 0) {
                    wait_bar(bar(C::bQF), q_use & 1, abort_flag, 2, C::bQF);
                    ++q_use;
                    for (int i = 0; i < no; ++i) {
                        const int s = it % C::kSlots;
                        wait_bar(bar(C::bF + s), (it / C::kSlots) & 1, abort_flag, 2, C::bF + s);
                        wait_bar(bar(C::bSE), (s_use & 1) ^ 1, abort_flag, 2, C::bSE);
                        tc_fence_after();
                        const uint64_t kd = rdesc0 + static_cast<uint64_t>((s * C::kTile) >> 4);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t off = static_cast<uint64_t>(((kk / 4) * 16384 + (kk % 4) * 32) >> 4);
                            tc_mma_f16(tmem + C::kColS, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(bar(C::bSF));
                        tc_commit(bar(C::bE + s));
                        ++it;
                        ++s_use;
                    }
                    tc_commit(bar(C::bQE));  // the Q tile, once the last Q K^T has read it
                }
                // the previous block's O has left TMEM before this block's P V (or,
                // with no tile here, its completion signal): bO never runs two
                // phases ahead of the workers
                if (k > 0) wait_bar(bar(C::bOE), (k - 1) & 1, abort_flag, 2, C::bOE);
                for (int i = 0; i < no; ++i) {
                    const int s = it % C::kSlots;
                    wait_bar(bar(C::bF + s), (it / C::kSlots) & 1, abort_flag, 2, C::bF + s);
                    wait_bar(bar(C::bPF + i), (pf_phase >> i) & 1, abort_flag, 2, C::bPF + i);
                    pf_phase ^= 1u << i;
                    tc_fence_after();
                    const uint64_t vd = vdesc0 + static_cast<uint64_t>((s * C::kTile) >> 4);
                    // O += P_i V_i: P from TMEM (keys 16 kk .. 16 kk + 15 in columns 8 kk ..)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_f16_ts(tmem + C::kColO, tmem + C::kColE + 64 * i + 8 * kk,
                                      vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar(C::bE + s));
                    ++it;
                }
                // every block, also one without tiles here: the workers wait for it
                tc_commit(bar(C::bO));
            }
        } else if (warp >= 2) {
            // ------------------------------------------------------------ causal zero tiles
            const int rb = row_begin((int)rank), re = row_begin((int)rank + 1);
            for (int k = 0;; ++k) {
                const int r = one_rank(k, cl, G);
                if (r >= n_items) break;
                const OneItem I = one_item(prm, r);
                const int r0 = I.qt * 128;
                zero_p_region(prm, I.b, I.h, r0 + rb, min(r0 + re, prm.Sq), I.n * 128, warp - 2, 2, lane);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax workers
        setmaxnreg_inc<kRegsHigh>();
        const int g = (warp - 4) >> 2;                      // warpgroup: keys [64 g, 64 g + 64) of a tile
        const int t = (threadIdx.x - 128) & 127;            // row within the block == TMEM lane
        const int wt = threadIdx.x - 128;                   // 0..255
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float cexp = kMasked ? 1.f : prm.c2;
        const int rb = row_begin((int)rank), re = row_begin((int)rank + 1);
        const int rows_max = (128 + CL - 1) / CL;
        const int owner = t * CL / 128;                     // CTA that reduces and stores row t of O
        const int own_slot_row = t - row_begin(owner);
        constexpr int kRowBytes = D * 4;
        const uint32_t box = sBox + (warp - 4) * C::kBoxBytes;
        int s_use = 0;
        if (lane == 0) prefetch_tmap(&tm_p);
        for (int k = 0;; ++k) {
            const int r = one_rank(k, cl, G);
            if (r >= n_items) break;
            const OneItem I = one_item(prm, r);
            const int no = n_own_of(I);
            const int r0 = I.qt * 128, row = r0 + t;
            const bool row_ok = row < prm.Sq;
            // bytes this block will receive (the peers cannot send them before this
            // CTA has finished the previous block: they need its statistics first)
            if (wt == 0) {
                mbar_arrive_expect_tx(bar(C::bST), (uint32_t)(CL * 128 * 8));
                mbar_arrive_expect_tx(bar(C::bRecv), (uint32_t)((CL - 1) * (re - rb) * kRowBytes));
            }

            // ---- A: S -> exponentials (fp16, TMEM) and the row's running (max, sum)
            float M = -CUDART_INF_F, L = 0.f;
            float mt[C::kMaxOwn];
#pragma unroll
            for (int i = 0; i < C::kMaxOwn; ++i) {
                mt[i] = -CUDART_INF_F;
                if (i < no) {
                    const int kv0 = ((int)rank + CL * i) * 128 + 64 * g;
                    wait_bar(bar(C::bSF), s_use & 1, abort_flag, 4, C::bSF);
                    tc_fence_after();
                    float s[64];
                    tmem_ld64(tmem + lane_base + C::kColS + 64 * g, s);
                    tc_fence_before();
                    mbar_arrive(bar(C::bSE));
                    ++s_use;
                    mask_tile<T, kMasked, 64>(s, prm, I.b, I.h, row, row_ok, kv0);
                    float mx[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) mx[x] = s[x];
#pragma unroll
                    for (int x = 8; x < 64; ++x) mx[x & 7] = fmaxf(mx[x & 7], s[x]);
                    const float m_t = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                            fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * cexp;
                    const float mm = m_t == -CUDART_INF_F ? 0.f : m_t;  // all masked: every e is 0
                    uint32_t hp[32];
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const float e0 = ex2(fmaf(s[2 * x], cexp, -mm));
                        const float e1 = ex2(fmaf(s[2 * x + 1], cexp, -mm));
                        acc[x & 3] += e0 + e1;
                        __half2 hh = __floats2half2_rn(e0, e1);
                        hp[x] = *reinterpret_cast<uint32_t*>(&hh);
                    }
                    tmem_st32(tmem + lane_base + C::kColE + 64 * i + 32 * g, hp);
                    if (m_t != -CUDART_INF_F) {
                        const float l_t = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                        const float Mn = fmaxf(M, m_t);
                        L = L * ex2(M - Mn) + l_t * ex2(m_t - Mn);
                        M = Mn;
                    }
                    mt[i] = m_t;
                }
            }

            // ---- B: the row LSE over the whole cluster.  The warpgroups merge
            // their (max, sum) here; warpgroup 0 sends the CTA's pair of every
            // row into every cluster CTA's statistics slots.
            if (g == 1) {
                mgM[t] = M;
                mgL[t] = L;
            }
            softmax_group_sync();
            if (g == 0) {
                const float M1 = mgM[t], L1 = mgL[t];
                const float Mc = fmaxf(M, M1);
                const float Lc = Mc == -CUDART_INF_F ? 0.f : L * ex2(M - Mc) + L1 * ex2(M1 - Mc);
                const uint32_t slot = sStat + (rank * 128 + t) * 8;
                for (int c = 0; c < CL; ++c)
                    st_async_v2(cluster_addr(slot, c), Mc, Lc, cluster_addr(bar(C::bST), c));
            }
            wait_bar_cluster(bar(C::bST), k & 1, abort_flag, 5, C::bST);
            float lse2;
            {
                const float2* st = reinterpret_cast<const float2*>(smem + C::kOffRecv + C::kRecvBytes - CL * 1024);
                float2 sv[kOneMaxCluster];
                float Mx = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < kOneMaxCluster; ++c) {
                    sv[c] = make_float2(-CUDART_INF_F, 0.f);
                    if (c < CL) {
                        sv[c] = st[c * 128 + t];
                        Mx = fmaxf(Mx, sv[c].x);
                    }
                }
                if (Mx == -CUDART_INF_F) {
                    lse2 = -CUDART_INF_F;
                } else {
                    float sum = 0.f;
#pragma unroll
                    for (int c = 0; c < kOneMaxCluster; ++c)
                        if (c < CL) sum += sv[c].y * ex2(sv[c].x - Mx);
                    lse2 = Mx + log2f(sum);
                }
            }
            const bool dead = lse2 == -CUDART_INF_F;

            // ---- C: P = e * exp2(m_j - lse): back into TMEM for P V, and through the
            // warp's swizzled box to a TMA store of P
#pragma unroll
            for (int i = 0; i < C::kMaxOwn; ++i) {
                if (i < no) {
                    const int kv0 = ((int)rank + CL * i) * 128 + 64 * g;
                    const float sc = (dead || mt[i] == -CUDART_INF_F) ? 0.f : ex2(mt[i] - lse2);
                    const uint32_t ecol = tmem + lane_base + C::kColE + 64 * i + 32 * g;
                    float ef[32];
                    tmem_ld32(ecol, ef);
                    uint32_t w[32];
                    if constexpr (kBF16) {
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const uint32_t bits = __float_as_uint(ef[x]);
                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&bits));
                            w[x] = Pack<T>::two(f.x * sc, f.y * sc);
                        }
                    } else {
                        // f16: one packed multiply per pair (e, the factor and the
                        // product each rounded to f16: at most 3 * 2^-12 relative)
                        const __half2 sc2 = __float2half2_rn(sc);
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const uint32_t bits = __float_as_uint(ef[x]);
                            __half2 hh = __hmul2(*reinterpret_cast<const __half2*>(&bits), sc2);
                            w[x] = *reinterpret_cast<uint32_t*>(&hh);
                        }
                    }
                    tmem_st32(ecol, w);
                    tc_fence_before();
                    mbar_arrive(bar(C::bPF + i));
                    // the box is free once this warp's previous P store has read it
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                    const uint32_t rowaddr = box + (t & 31) * 128;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(rowaddr + ((u ^ (t & 7)) * 16), w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int prow = r0 + 32 * (warp & 3);
                        tma_store_4d(&tm_p, box, kv0, pick(prm.ord_p & 3, prow, I.h, I.b),
                                     pick((prm.ord_p >> 2) & 3, prow, I.h, I.b),
                                     pick((prm.ord_p >> 4) & 3, prow, I.h, I.b));
                        bulk_commit();
                    }
                }
            }

            // ---- D: partial O rows to their owners (st.async, 16-byte units of row
            // t at unit ^ (t % 8)); this CTA adds the peers' rows to its own
            wait_bar(bar(C::bO), k & 1, abort_flag, 6, C::bO);
            tc_fence_after();
            float ov[D / 2];
            if (no > 0) {
                if constexpr (D == 128) tmem_ld64(tmem + lane_base + C::kColO + g * 64, ov);
                else tmem_ld32(tmem + lane_base + C::kColO + g * 32, ov);
            } else {
#pragma unroll
                for (int x = 0; x < D / 2; ++x) ov[x] = 0.f;
            }
            tc_fence_before();
            softmax_group_sync();  // O is out of TMEM
            if (wt == 0) mbar_arrive(bar(C::bOE));
            if (owner != (int)rank) {
                const int slot = (int)rank < owner ? (int)rank : (int)rank - 1;
                const uint32_t dst = cluster_addr(sRecv + (slot * rows_max + own_slot_row) * kRowBytes, owner);
                const uint32_t rbar = cluster_addr(bar(C::bRecv), owner);
#pragma unroll
                for (int u = 0; u < D / 8; ++u) {
                    const int pu = (g * (D / 8) + u) ^ (t & 7);
                    st_async_v4(dst + pu * 16, __float_as_uint(ov[4 * u]), __float_as_uint(ov[4 * u + 1]),
                                __float_as_uint(ov[4 * u + 2]), __float_as_uint(ov[4 * u + 3]), rbar);
                }
            }
            wait_bar_cluster(bar(C::bRecv), k & 1, abort_flag, 6, C::bRecv);
            if (owner == (int)rank) {
#pragma unroll
                for (int sl = 0; sl < kOneMaxCluster - 1; ++sl) {
                    if (sl < CL - 1) {
                        const uint32_t src = sRecv + (sl * rows_max + own_slot_row) * kRowBytes;
#pragma unroll
                        for (int u = 0; u < D / 8; ++u) {
                            const int pu = (g * (D / 8) + u) ^ (t & 7);
                            const uint4 a = ld_shared_v4(src + pu * 16);
                            ov[4 * u] += __uint_as_float(a.x);
                            ov[4 * u + 1] += __uint_as_float(a.y);
                            ov[4 * u + 2] += __uint_as_float(a.z);
                            ov[4 * u + 3] += __uint_as_float(a.w);
                        }
                    }
                }
                if (row_ok) {
                    T* op = static_cast<T*>(prm.o) + I.b * prm.so0 + I.h * prm.so1 + (long long)row * prm.so2 + g * (D / 2);
#pragma unroll
                    for (int u = 0; u < D / 16; ++u) {
                        uint4 w4;
                        w4.x = Pack<T>::two(ov[8 * u], ov[8 * u + 1]);
                        w4.y = Pack<T>::two(ov[8 * u + 2], ov[8 * u + 3]);
                        w4.z = Pack<T>::two(ov[8 * u + 4], ov[8 * u + 5]);
                        w4.w = Pack<T>::two(ov[8 * u + 6], ov[8 * u + 7]);
                        reinterpret_cast<uint4*>(op)[u] = w4;
                    }
                }
            }
            if (rank == 0 && g == 0 && prm.lse && row_ok)
                prm.lse[((long long)I.b * prm.Hq + I.h) * prm.Sq + row] = dead ? lse2 : lse2 * kLn2;
            softmax_group_sync();  // the receive area is read before this CTA's statistics of the next block go out
        }
        if (lane == 0) bulk_wait0();
    }

    // ------------------------------------------------------------ teardown
    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // no CTA leaves while a peer may still write into its shared memory
    if (warp == 1) {
        tc_fence_after();
        if (*abort_flag) {
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        }
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- fused single-sweep kernel
// Row blocks with at most two live 128-key score tiles (Skv <= 256, or a
// causal mask over at most 256 query rows): S for every live key of the row
// block stays in TMEM, so the row max, the sum of exponentials and
// P = exp(S - lse) all come from one Q K^T, and the whole forward is one
// launch with no second sweep (the small-shape fused variant of the page's
// "single-kernel fusion (small shapes)" update, which counts tiles after
// causal truncation).  Keys past the live tiles get P = 0.
//
// One CTA (256 threads, two warpgroups) per 128-row query tile of one
// (batch, head).  Q, K and V arrive by asynchronous 16-byte copies straight in
// the 128B-swizzled operand layout (any row stride that keeps rows 16-byte
// aligned); a bool mask tile is staged in shared memory with coalesced loads;
// warpgroup w owns key tile w.  P goes to the swizzled A-operand tile of P V,
// from which warps copy it to global memory row by row with coalesced stores
// that follow the alignment of the caller's P rows (a 100-key row of 200 bytes
// is fine).  Every wait is bounded.
struct FusedIO {
    const void* q; long long sq0, sq1, sq2;
    const void* k; long long sk0, sk1, sk2;
    const void* v; long long sv0, sv1, sv2;
    uint32_t tmem_cols;  // power of two >= S columns + D
    int rpc;             // query rows per CTA: 128, or 32 to spread a small grid over more SMs
};

struct FusedCfg {
    static constexpr int kThreads = 256;
    static constexpr int kMaxKeyTiles = 2;
};

template <int D>
struct FusedSmem {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTile;
    static constexpr int kOffV = kOffK + FusedCfg::kMaxKeyTiles * kTile;
    static constexpr int kOffP = kOffV + FusedCfg::kMaxKeyTiles * kTile;
    static constexpr int kEnd = kOffP + FusedCfg::kMaxKeyTiles * 128 * 128 * 2;
    // float[2 (max, sum)][2 warpgroups][128]; aliases K, which is dead once S is in TMEM
    static constexpr int kOffStat = kOffK;
    // bool mask tile [128 rows][kMaskPitch bytes] (odd word pitch: conflict-free
    // row-per-thread reads); after the statistics in the dead K tiles when they
    // have room, else in its own region
    static constexpr int kMaskPitch = 260;
    static constexpr int kMaskBytes = 128 * kMaskPitch;
    static constexpr bool kMaskInK = 2048 + kMaskBytes <= FusedCfg::kMaxKeyTiles * kTile;
    static constexpr int kOffMask = kMaskInK ? kOffK + 2048 : kEnd;
    static constexpr int kOffBar = kMaskInK ? kEnd : kEnd + kMaskBytes;
    static constexpr int kSmem = kOffBar + 64 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// Rows [0, nvalid) of a [rows, X] slice (element row stride srow, rows
// 16-byte aligned) into a 128-row 128B-swizzled tile with asynchronous 16-byte
// copies (all in flight together); rows past nvalid are zero-filled.
template <typename T>
__device__ __forceinline__ void load_tile_sw128(uint32_t dst, const T* src, long long srow, int nvalid, int X) {
    const int upr = X / 8;  // 16-byte units per row
    for (int u = threadIdx.x; u < 128 * upr; u += FusedCfg::kThreads) {
        const int r = u / upr, c = u % upr;
        const bool ok = r < nvalid;
        const T* g = ok ? src + r * srow + c * 8 : src;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                         dst + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4)),
                     "l"(g), "r"(ok ? 16 : 0)
                     : "memory");
    }
}

template <int D, typename T, bool kMasked>
__global__ void __launch_bounds__(FusedCfg::kThreads, 1)
tc_fused_kernel(const TcParams prm, const FusedIO io) {
    using L = FusedSmem<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sQ = smem_u32(smem + L::kOffQ), sK = smem_u32(smem + L::kOffK);
    const uint32_t sV = smem_u32(smem + L::kOffV), sP = smem_u32(smem + L::kOffP);
    float* stat = reinterpret_cast<float*>(smem + L::kOffStat);  // [2 (max, sum)][2 warpgroups][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // [0] S ready, [1] O ready
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.x, b = blockIdx.y, qt = blockIdx.z;
    const int hk = h / prm.group;
    const int r0 = qt * io.rpc;
    const int r_end = min(r0 + io.rpc, prm.Sq);  // this CTA's rows are [r0, r_end)
    // live key tiles of this row block (1 or 2): with a causal mask the keys
    // past its last row are masked for every row, so they are never computed
    // and their P columns are written as zeros
    int n_kv = (prm.Skv + 127) / 128;
    if (prm.causal) n_kv = min(n_kv, min(r_end - 1, prm.Skv - 1) / 128 + 1);
    const int live_end = min(prm.Skv, n_kv * 128);  // keys [live_end, Skv) have P = 0 in every row
    const uint32_t kTmemO = n_kv * 128;             // O columns follow the S tiles

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), io.tmem_cols);
        tmem_relinquish();
    }
    // Q tile, K and V tiles -> swizzled operand tiles
    const T* Q = static_cast<const T*>(io.q) + b * io.sq0 + h * io.sq1 + (long long)r0 * io.sq2;
    load_tile_sw128<T>(sQ, Q, io.sq2, r_end - r0, D);
    for (int j = 0; j < n_kv; ++j) {
        const T* K = static_cast<const T*>(io.k) + b * io.sk0 + hk * io.sk1 + (long long)(j * 128) * io.sk2;
        const T* V = static_cast<const T*>(io.v) + b * io.sv0 + hk * io.sv1 + (long long)(j * 128) * io.sv2;
        const int nv = min(128, prm.Skv - j * 128);
        load_tile_sw128<T>(sK + j * L::kTile, K, io.sk2, nv, D);
        load_tile_sw128<T>(sV + j * L::kTile, V, io.sv2, nv, D);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // A bool mask is read once per CTA with coalesced loads (warp w takes rows
    // w, w+8, ...; lanes take consecutive 4-byte words, or bytes when the rows
    // are not 4-byte aligned) while the tiles are in flight, and staged in
    // shared memory once S is ready (the staging area may alias K).
    constexpr int kMaskRowsPerWarp = 16;
    uint32_t mreg[kMaskRowsPerWarp][2];
    const bool stage_mask = kMasked && prm.mask_kind == kMaskBool;
    const unsigned char* mbase = static_cast<const unsigned char*>(prm.mask) + b * prm.sm0 + h * prm.sm1;
    const bool m_words = stage_mask && ((reinterpret_cast<uintptr_t>(mbase) | (uintptr_t)prm.sm2) & 3) == 0;
    if (stage_mask) {
#pragma unroll
        for (int i = 0; i < kMaskRowsPerWarp; ++i) {
            const int rr = warp + 8 * i, grow = r0 + rr;
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {
                uint32_t v = 0;
                if (grow < r_end) {
                    const unsigned char* mr = mbase + (long long)grow * prm.sm2;
                    if (m_words) {
                        const int k4 = 4 * (lane + 32 * hw);
                        if (k4 + 4 <= prm.Skv) v = *reinterpret_cast<const uint32_t*>(mr + k4);
                        else
                            for (int e = 0; e < 4; ++e)
                                if (k4 + e < prm.Skv) v |= static_cast<uint32_t>(mr[k4 + e]) << (8 * e);
                    } else {
                        const int k1 = lane + 32 * hw;  // bytes: keys k1, k1 + 64, k1 + 128, k1 + 192
                        for (int e = 0; e < 4; ++e)
                            if (k1 + 64 * e < prm.Skv) v |= static_cast<uint32_t>(mr[k1 + 64 * e]) << (8 * e);
                    }
                }
                mreg[i][hw] = v;
            }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // S_j = Q K_j^T for both key tiles, one commit
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBF16, false);
        for (int j = 0; j < n_kv; ++j)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                tc_mma_f16(tmem + j * 128, sw128_desc(sQ + off, 16, 1024),
                           sw128_desc(sK + j * L::kTile + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
            }
        tc_commit(smem_u32(&bars[0]));
    }

    // warpgroup g takes keys [64 g, 64 g + 64) of every live tile, row t
    const int wg = threadIdx.x / 128, t = threadIdx.x % 128;
    const int row = r0 + t;
    const bool row_ok = row < r_end;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float cexp = kMasked ? 1.f : prm.c2;
    wait_bar(smem_u32(&bars[0]), 0, abort_flag, 7, 0);
    tc_fence_after();
    const uint32_t sMask = smem_u32(smem + L::kOffMask);
    if (stage_mask) {
#pragma unroll
        for (int i = 0; i < kMaskRowsPerWarp; ++i) {
            const int rr = warp + 8 * i;
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {
                const uint32_t v = mreg[i][hw];
                if (m_words) {
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(sMask + rr * L::kMaskPitch + 4 * (lane + 32 * hw)), "r"(v)
                                 : "memory");
                } else {
                    const int k1 = lane + 32 * hw;
                    for (int e = 0; e < 4; ++e)
                        asm volatile("st.shared.u8 [%0], %1;" ::"r"(sMask + rr * L::kMaskPitch + k1 + 64 * e),
                                     "r"((v >> (8 * e)) & 0xffu)
                                     : "memory");
                }
            }
        }
        __syncthreads();
    }
    float s[FusedCfg::kMaxKeyTiles][64];
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < FusedCfg::kMaxKeyTiles; ++j) {
        if (j < n_kv) {
            const int kv0 = j * 128 + 64 * wg;
            tmem_ld64(tmem + lane_base + j * 128 + 64 * wg, s[j]);
            if (stage_mask) {
                // keys of this row from the staged tile (zero bytes past Skv / Sq)
                const uint32_t mrow = sMask + t * L::kMaskPitch + kv0;
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    uint32_t m4;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(m4) : "r"(mrow + 4 * w));
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        s[j][4 * w + e] = ((m4 >> (8 * e)) & 0xffu) ? fmaf(s[j][4 * w + e], prm.c2, 0.f) : -CUDART_INF_F;
                }
                mask_tile<T, false, 64>(s[j], prm, b, h, row, row_ok, kv0);  // ragged keys / rows
            } else {
                mask_tile<T, kMasked, 64>(s[j], prm, b, h, row, row_ok, kv0);
            }
#pragma unroll
            for (int x = 0; x < 64; ++x) mt = fmaxf(mt, s[j][x]);
        }
    }
    stat[wg * 128 + t] = mt * cexp;
    __syncthreads();
    const float m = fmaxf(stat[t], stat[128 + t]);
    float lpart = 0.f;
    if (m != -CUDART_INF_F) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < FusedCfg::kMaxKeyTiles; ++j)
            if (j < n_kv) {
#pragma unroll
                for (int x = 0; x < 64; ++x) acc[x & 7] += ex2(fmaf(s[j][x], cexp, -m));
            }
        lpart = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    }
    stat[256 + wg * 128 + t] = lpart;
    __syncthreads();
    const float l = stat[256 + t] + stat[384 + t];
    const float lse2 = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
    const bool dead = lse2 == -CUDART_INF_F;
    const float neg = dead ? -CUDART_INF_F : -lse2;
#pragma unroll
    for (int j = 0; j < FusedCfg::kMaxKeyTiles; ++j) {
        if (j < n_kv) {
            uint32_t hp[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                hp[x] = Pack<T>::two(ex2(fmaf(s[j][2 * x], cexp, neg)), ex2(fmaf(s[j][2 * x + 1], cexp, neg)));
            // chunk wg of P tile j, row t (16-byte unit u at u ^ (t % 8))
            const uint32_t rowaddr = sP + j * 128 * 128 * 2 + wg * 16384 + t * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                st_shared_v4(rowaddr + ((u ^ (t & 7)) * 16), hp[4 * u], hp[4 * u + 1], hp[4 * u + 2], hp[4 * u + 3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
        tc_fence_after();
        constexpr uint32_t idesc_pv = idesc_f16(128, D, kBF16, true);
        for (int j = 0; j < n_kv; ++j)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a_off = (kk / 4) * 16384 + (kk % 4) * 32;
                const uint32_t b_off = kk * 2048;
                tc_mma_f16(tmem + kTmemO, sw128_desc(sP + j * 128 * 128 * 2 + a_off, 16, 1024),
                           sw128_desc(sV + j * L::kTile + b_off, 16384, 1024), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            }
        tc_commit(smem_u32(&bars[1]));
    }
    // P rows to global memory while P V runs
    {
        const int nrows = r_end - r0;
        // shared address of P[rr, key] (key < live_end)
        auto src = [&](int rr, int key) {
            const int kt = key & 127;
            return sP + (key >> 7) * (128 * 128 * 2) + (kt >> 6) * 16384 + rr * 128 +
                   ((((kt >> 3) & 7) ^ (rr & 7)) << 4) + (kt & 7) * 2;
        };
        uint16_t* pslab = static_cast<uint16_t*>(prm.p) + b * prm.sp0 + h * prm.sp1 + (long long)r0 * prm.sp2;
        {
            // row by row: warp w copies rows w, w+8, ...; lanes take consecutive
            // key pairs (4-byte stores) or, with only 2-byte aligned rows, keys
            for (int rr = warp; rr < nrows; rr += 8) {
                uint16_t* prow = pslab + (long long)rr * prm.sp2;
                // (live_end is a multiple of 128 or Skv, so a key pair never straddles it)
                if ((reinterpret_cast<uintptr_t>(prow) & 3) == 0) {
                    for (int key = 2 * lane; key < prm.Skv; key += 64) {
                        uint32_t v = 0;
                        if (key < live_end) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(src(rr, key)));
                        if (key + 1 < prm.Skv) *reinterpret_cast<uint32_t*>(prow + key) = v;
                        else prow[key] = static_cast<uint16_t>(v);
                    }
                } else {
                    for (int key = lane; key < prm.Skv; key += 32) {
                        uint16_t v = 0;
                        if (key < live_end) asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(src(rr, key)));
                        prow[key] = v;
                    }
                }
            }
        }
    }
    wait_bar(smem_u32(&bars[1]), 0, abort_flag, 7, 1);
    tc_fence_after();
    // O: warpgroup w writes columns [w D/2, (w+1) D/2) of its rows
    {
        T* orow = static_cast<T*>(prm.o) + b * prm.so0 + h * prm.so1 + (long long)row * prm.so2 + wg * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            float ov[32];
            tmem_ld32(tmem + lane_base + kTmemO + wg * (D / 2) + c * 32, ov);
            if (row_ok) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 pk;
                    pk.x = Pack<T>::two(dead ? 0.f : ov[u * 8 + 0], dead ? 0.f : ov[u * 8 + 1]);
                    pk.y = Pack<T>::two(dead ? 0.f : ov[u * 8 + 2], dead ? 0.f : ov[u * 8 + 3]);
                    pk.z = Pack<T>::two(dead ? 0.f : ov[u * 8 + 4], dead ? 0.f : ov[u * 8 + 5]);
                    pk.w = Pack<T>::two(dead ? 0.f : ov[u * 8 + 6], dead ? 0.f : ov[u * 8 + 7]);
                    *reinterpret_cast<uint4*>(orow + c * 32 + u * 8) = pk;
                }
            }
        }
    }
    if (wg == 0 && prm.lse && row_ok)
        prm.lse[((long long)b * prm.Hq + h) * prm.Sq + row] = dead ? lse2 : lse2 * kLn2;

    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (*abort_flag)
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        tmem_dealloc(tmem, io.tmem_cols);
    }
}


// ---------------------------------------------------------------- tensor-core decode / split-KV
//
// Few query rows per key/value head (R = group * Sq <= 16), any number of keys,
// D = Dv = 128.  One cluster of C CTAs per (batch, key/value head); CTA c owns
// a contiguous chunk of keys, walked in 128-key tiles.  The dot products run
// on the tensor cores with the keys on the TMEM lanes:
//   sweep 1: S^T = K_tile Q^T (M = 128 keys, N = 16 query rows, zero-padded),
//     so thread t reads key t's R scores with one tcgen05.ld; the scores of the
//     chunk stay in shared memory;
//   the chunk statistics are merged over the cluster through DSMEM (every CTA
//     forms the same lse per row);
//   sweep 2: P = exp2(s - lse) per (row, key), stored to global memory and as
//     the B operand of O^T += V_tile^T P^T (M = 128 value columns, A read
//     MN-major from the V tile as loaded);
//   the partial O^T is summed over the cluster by column slices.
// K and V tiles arrive by TMA through one ring shared by both sweeps.

struct TcDecParams {
    const void* q; long long sq0, sq1, sq2;
    const void* mask; int mask_kind, mask_dtype; long long sm0, sm1, sm2;
    void* o; long long so0, so1, so2;
    void* p; long long sp0, sp1, sp2;
    float* lse;
    int Hq, Sq, Skv, group, rows, chunk, causal, stages;
    float c2;  // scale * log2(e)
    uint32_t ord_k, ord_v;
    int off_ss, off_part, off_st;  // dynamic shared-memory layout after the fixed part
};

constexpr int kDecThreads = 128;
constexpr int kDecMaxCluster = 16;
constexpr int kDecSmemMax = 220 * 1024;  // dynamic shared memory (the kernel also has a little static)
struct DecLayout {
    static constexpr int kTile = 128 * 128 * 2;         // one K or V tile
    static constexpr int kMaxStages = 3;                // the ring starts at offset 0
    static constexpr int kOffQ = kMaxStages * kTile;     // [16 rows, 128] K-major
    static constexpr int kOffP = kOffQ + 4096;           // two [16 rows, 128 keys] P^T operands
    static constexpr int kOffBar = kOffP + 8192;
    static constexpr int kFixed = kOffBar + 128;
    // the ring is placed for kMaxStages; a two-stage launch moves everything after it down
    static constexpr int kRingShrink2 = kTile;
};

template <typename T>
__global__ void __launch_bounds__(kDecThreads, 1)
tc_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const TcDecParams p) {
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kCols = 64;  // S^T [0, 32) double-buffered, O^T [32, 48)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ float lse_s[16];
    __shared__ int row_h[16], row_i[16];
    const int shrink = p.stages == 2 ? DecLayout::kRingShrink2 : 0;
    const uint32_t sRing = smem_u32(smem);
    const uint32_t sQ = smem_u32(smem + DecLayout::kOffQ - shrink), sP = smem_u32(smem + DecLayout::kOffP - shrink);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DecLayout::kOffBar - shrink);  // full[3], s[2], o
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* ss = reinterpret_cast<float*>(smem + p.off_ss);      // [R][chunk] scores, base-2 units
    float* part = reinterpret_cast<float*>(smem + p.off_part);  // [R][128] partial O
    float* st = reinterpret_cast<float*>(smem + p.off_st);      // [R][2] chunk (max, sum)
    auto bar_full = [&](int s) { return smem_u32(&bars[s]); };
    auto bar_s = [&](int i) { return smem_u32(&bars[3 + (i & 1)]); };
    const uint32_t bar_o = smem_u32(&bars[5]);

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const uint32_t crank = cluster_ctarank();
    const int C = (int)gridDim.x;
    const int b = blockIdx.z, hk = blockIdx.y;
    const int k0 = (int)crank * p.chunk;
    const int n = max(0, min(p.Skv, k0 + p.chunk) - k0);
    const int nt = (n + 127) / 128;
    const int R = p.rows, S = p.stages;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    if (t == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(smem_u32(&bars[i]), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kCols);
        tmem_relinquish();
    }
    // Q rows (zero rows past R) in the swizzled K-major layout; P^T operands zeroed
    for (int u = t; u < 16 * 16; u += kDecThreads) {
        const int r = u / 16, c = u % 16;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < R) {
            const T* qr = static_cast<const T*>(p.q) + b * p.sq0 + (long long)(hk * p.group + r / p.Sq) * p.sq1 +
                          (long long)(r % p.Sq) * p.sq2;
            v = *reinterpret_cast<const uint4*>(qr + c * 8);
        }
        st_shared_v4(sQ + (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4), v.x, v.y, v.z, v.w);
    }
    for (int u = t; u < 8192 / 16; u += kDecThreads) st_shared_v4(sP + 16 * u, 0u, 0u, 0u, 0u);
    if (t < R) {
        row_h[t] = hk * p.group + t / p.Sq;
        row_i[t] = t % p.Sq;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ring uses: K tiles 0 .. nt-1, then V tiles 0 .. nt-1 (thread 0 issues)
    auto issue = [&](int use) {
        if (use >= 2 * nt) return;
        const bool is_v = use >= nt;
        const int i = is_v ? use - nt : use, row0 = k0 + i * 128;
        const int slot = use % S;
        const CUtensorMap* tm = is_v ? &tm_v : &tm_k;
        const uint32_t ord = is_v ? p.ord_v : p.ord_k;
        mbar_arrive_expect_tx(bar_full(slot), DecLayout::kTile);
        for (int c = 0; c < 2; ++c)
            tma_load_4d(sRing + slot * DecLayout::kTile + c * 16384, tm, bar_full(slot), c * 64,
                        pick(ord & 3, row0, hk, b), pick((ord >> 2) & 3, row0, hk, b), pick((ord >> 4) & 3, row0, hk, b));
    };
    if (t == 0)
        for (int u = 0; u < S; ++u) issue(u);
    constexpr uint32_t idesc_s = idesc_f16(128, 16, kBF16, false);
    constexpr uint32_t idesc_o = idesc_f16(128, 16, kBF16, false) | (1u << 15);  // A (V^T) MN-major

    // ---- sweep 1: scores
    for (int i = 0; i < nt; ++i) {
        const int slot = i % S;
        const uint32_t sK = sRing + slot * DecLayout::kTile;
        if (t == 0) {
            wait_bar(bar_full(slot), (i / S) & 1, abort_flag, 10, 0);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16(tmem + (i & 1) * 16, sw128_desc(sK + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                           sw128_desc(sQ + (kk / 4) * 2048 + (kk % 4) * 32, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            tc_commit(bar_s(i));
        }
        wait_bar(bar_s(i), (i >> 1) & 1, abort_flag, 10, 1);
        tc_fence_after();
        float acc[16];
        tmem_ld16(tmem + lane_base + (i & 1) * 16, acc);
        const int j = i * 128 + t, key = k0 + j;
        if (j < n) {
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < R) {
                    float sc = __fmul_rn(acc[r], p.c2);
                    if (p.causal && key > row_i[r]) sc = -CUDART_INF_F;
                    if (p.mask_kind != kMaskNone) {
                        const long long off = b * p.sm0 + row_h[r] * p.sm1 + (long long)row_i[r] * p.sm2 + key;
                        if (p.mask_kind == kMaskBool) {
                            if (static_cast<const unsigned char*>(p.mask)[off] == 0) sc = -CUDART_INF_F;
                        } else {
                            const float m = p.mask_dtype == kF32 ? static_cast<const float*>(p.mask)[off]
                                                                 : Pack<T>::load(static_cast<const T*>(p.mask) + off);
                            sc = __fmaf_rn(m, kLog2e, sc);
                        }
                    }
                    ss[r * p.chunk + j] = sc;
                }
        }
        tc_fence_before();
        __syncthreads();  // S^T buffer and the K tile consumed
        if (t == 0) issue(i + S);
    }

    // per-row (max, sum of exp2) of the chunk: one warp per row
    for (int r = warp; r < R; r += kDecThreads / 32) {
        float m = -CUDART_INF_F;
        for (int j = lane; j < n; j += 32) m = fmaxf(m, ss[r * p.chunk + j]);
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        if (m != -CUDART_INF_F)
            for (int j = lane; j < n; j += 32) l += exp2f(ss[r * p.chunk + j] - m);
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            st[2 * r] = m;
            st[2 * r + 1] = l;
        }
    }
    // ---- the cluster's statistics -> the same lse in every CTA
    cluster_barrier();
    if (t < R) {
        float mc[kDecMaxCluster], lc[kDecMaxCluster];
#pragma unroll
        for (int c = 0; c < kDecMaxCluster; ++c)
            if (c < C) {
                mc[c] = ld_cluster_f32(&st[2 * t], (uint32_t)c);
                lc[c] = ld_cluster_f32(&st[2 * t + 1], (uint32_t)c);
            }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < kDecMaxCluster; ++c)
            if (c < C) m = fmaxf(m, mc[c]);
        float l = 0.f;
        if (m != -CUDART_INF_F) {
#pragma unroll
            for (int c = 0; c < kDecMaxCluster; ++c)
                if (c < C && mc[c] != -CUDART_INF_F) l += lc[c] * exp2f(mc[c] - m);
        }
        lse_s[t] = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
    }
    __syncthreads();

    // ---- sweep 2: P (stored, and as the rounded B operand), O^T += V^T P^T
    for (int i = 0; i < nt; ++i) {
        const int use = nt + i, slot = use % S;
        const uint32_t sV = sRing + slot * DecLayout::kTile, sPb = sP + (i & 1) * 4096;
        const int j = i * 128 + t;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r < R) {
                const float L = lse_s[r];
                const float pr = (j < n && L != -CUDART_INF_F) ? exp2f(ss[r * p.chunk + j] - L) : 0.f;
                const T pt = from_float<T>(pr);
                if (j < n) {
                    T* prow = static_cast<T*>(p.p) + b * p.sp0 + row_h[r] * p.sp1 + (long long)row_i[r] * p.sp2;
                    prow[k0 + j] = pt;
                }
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(sPb + (t >> 6) * 2048 + r * 128 +
                                                             ((((t & 63) >> 3) ^ (r & 7)) << 4) + (t & 7) * 2),
                             "h"(bits16(pt))
                             : "memory");
            }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (t == 0) {
            tc_fence_after();
            wait_bar(bar_full(slot), (use / S) & 1, abort_flag, 10, 2);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16(tmem + 32, sw128_desc(sV + kk * 2048, 16384, 1024),
                           sw128_desc(sPb + (kk / 4) * 2048 + (kk % 4) * 32, 16, 1024), idesc_o,
                           (i > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_o);
            wait_bar(bar_o, i & 1, abort_flag, 10, 3);  // the V tile and this P^T buffer are free again
            issue(use + S);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- partial O (lane t = value column t), then the cluster sum by column slices
    {
        float o[16];
        tmem_ld16(tmem + lane_base + 32, o);
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r < R) part[r * 128 + t] = nt > 0 ? o[r] : 0.f;
    }
    cluster_barrier();
    const int cols = (128 + C - 1) / C;
    const int c0 = (int)crank * cols, c1 = min(128, c0 + cols);
    for (int e = t; e < R * max(0, c1 - c0); e += kDecThreads) {
        const int r = e / (c1 - c0), d = c0 + e % (c1 - c0);
        float pc[kDecMaxCluster];
#pragma unroll
        for (int c = 0; c < kDecMaxCluster; ++c)
            if (c < C) pc[c] = ld_cluster_f32(&part[r * 128 + d], (uint32_t)c);
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kDecMaxCluster; ++c)
            if (c < C) acc += pc[c];
        const bool dead = lse_s[r] == -CUDART_INF_F;
        T* orow = static_cast<T*>(p.o) + b * p.so0 + row_h[r] * p.so1 + (long long)row_i[r] * p.so2;
        orow[d] = from_float<T>(dead ? 0.f : acc);
    }
    if (crank == 0 && p.lse && t < R) {
        const float L = lse_s[t];
        p.lse[((long long)b * p.Hq + row_h[t]) * p.Sq + row_i[t]] = (L == -CUDART_INF_F) ? L : L * kLn2;
    }
    __syncwarp();  // each warp reaches the cluster-wide barrier converged: lane-0 roles end later than their warp
    cluster_barrier();  // no CTA leaves while a peer may still read its shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (*abort_flag)
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        tmem_dealloc(tmem, kCols);
    }
}

// ---------------------------------------------------------------- backward
//
// Gradients of the (O, P) forward for dout (of O) and dprobs (of P) given P
// (FlagOS-OP PR #10, A1 item and the "P800 fused backward" update):
//   dP = dO V^T + dprobs,  r = rowsum(P * dP),  dS = P * (dP - r),
//   dQ = scale dS K,  dK = scale sum_h dS^T Q,  dV = sum_h P^T dO
// (sums over the query heads of a key/value head).  Every product is a
// tcgen05 MMA with fp32 accumulation in TMEM.
//   rows kernel: CTA per 128-row query tile of one head, one sweep over the
//     keys in 64-key steps: r and dQ through E = P * (dP + dprobs) (see the
//     kernel).  Writes dQ and r (the caller's row buffer).
//   keys kernel: CTA per 128-key tile of one key/value head, stepping over the
//     group's query heads in 64-row query tiles: dP^T (lanes = keys), dS^T
//     rounded to the input type, dV += P^T dO and dK += dS^T Q, accumulated
//     over the whole group in TMEM.
// Operands are staged with asynchronous 16-byte copies into 128-byte-swizzled
// tiles through multi-stage rings; a [query][key] tile (P, dprobs) serves as a
// K-major A operand (keys = K) and as an MN-major one (keys = M).  Separate
// mbarriers for the two MMA groups of a step let the second group of one step
// run under the start of the next.  Only D == Dv in {64, 128} and 16-byte
// aligned rows.

struct BwdIO {
    const void* q; long long sq0, sq1, sq2;
    const void* k; long long sk0, sk1, sk2;
    const void* v; long long sv0, sv1, sv2;
    const void* p; long long sp0, sp1, sp2;
    const void* go; long long sgo0, sgo1, sgo2;
    const void* gp; long long sgp0, sgp1, sgp2;  // dprobs, or null
    void* dq; long long sdq0, sdq1, sdq2;
    void* dk; long long sdk0, sdk1, sdk2;
    void* dv; long long sdv0, sdv1, sdv2;
    float* rowsum;  // [B, Hq, Sq] contiguous
    int Hq, group, Sq, Skv;
    float scale;
};

constexpr int kBwdThreads = 256;  // two warpgroups: the same 128 TMEM lanes, two column halves


// 16-byte chunk c (keys 8c .. 8c+7) of row r of a swizzled [128, 128] tile.
__device__ __forceinline__ uint32_t sw_chunk(uint32_t tile, int r, int c) {
    return tile + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}


__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
}

template <typename T> __device__ __forceinline__ float2 unpack_pair(uint32_t w);
template <> __device__ __forceinline__ float2 unpack_pair<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<__half2*>(&w));
}
template <> __device__ __forceinline__ float2 unpack_pair<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
}


// Rows kernel layout: dO once, then a three-stage ring of 64-key steps
// (V_j K-major, K_j MN-major, P_ij and dprobs_ij; E hi / lo overwrite the last two).
template <int D>
struct BwdRowsSmem {
    static constexpr int kStages = 3;
    static constexpr int kKeys = 64;
    static constexpr int kKV = kKeys * D * 2;     // [64, D] tile
    static constexpr int kPG = 128 * kKeys * 2;   // [128, 64] tile
    static constexpr int kStage = 2 * kKV + 2 * kPG;
    static constexpr int kOffDO = 0;
    static constexpr int kOffRing = 128 * D * 2;
    static constexpr int kOffStat = kOffRing + kStages * kStage;
    static constexpr int kOffBar = kOffStat + 1024;
    static constexpr int kSmem = kOffBar + 64 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert(kKV % 1024 == 0 && kPG % 1024 == 0, "tiles on 1024-byte boundaries");
};

// One sweep over the keys.  With E = P * (dP + dprobs) (fp32),
//   r = rowsum(E),  dQ = scale (sum_j E_j K_j - r sum_j P_j K_j),
// which equals scale * dS K without knowing r during the sweep.  E enters the
// MMA as two rounded parts, E_hi = rn(E) and E_lo = rn(E - E_hi), so the
// product is accurate to about fp32 and the final subtraction loses nothing
// beyond fp32 rounding.  TMEM: dP [0, 64), A = sum E K [64, 64 + D),
// Bp = sum P K [64 + D, 64 + 2D).
// Tensor-map order codes (see pick()) of the backward's TMA operands.
struct BwdOrd {
    uint32_t go, v, k, q, p, g;
};

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_tc_rows_kernel(const __grid_constant__ CUtensorMap tm_go, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_p,
                   const __grid_constant__ CUtensorMap tm_g, const BwdIO io, const BwdOrd ord) {
    using L = BwdRowsSmem<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kCols = 64 + 2 * D <= 256 ? 256 : 512;
    constexpr uint32_t tA = 64, tB = 64 + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sDO = smem_u32(smem + L::kOffDO), sRing = smem_u32(smem + L::kOffRing);
    float* stat = reinterpret_cast<float*>(smem + L::kOffStat);  // [2 warpgroups][128] partial row sums
    // [0] dP and Bp done, [1] A done, [2 + stage] stage loaded
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 + L::kStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, wg = threadIdx.x / 128, t = threadIdx.x % 128;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / io.group, r0 = qt * 128;
    const int nrows = min(128, io.Sq - r0);
    const int nsteps = (io.Skv + L::kKeys - 1) / L::kKeys;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t bar_dp = smem_u32(&bars[0]), bar_a = smem_u32(&bars[1]);
    auto bar_full = [&](int st) { return smem_u32(&bars[2 + st]); };
    const bool has_g = io.gp != nullptr;

    if (threadIdx.x == 0) {
        mbar_init(bar_dp, 1);
        mbar_init(bar_a, 1);
        for (int st = 0; st < L::kStages; ++st) mbar_init(bar_full(st), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_go);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_p);
        if (has_g) prefetch_tmap(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kCols);
        tmem_relinquish();
    }
    auto stage_v = [&](int st) { return sRing + st * L::kStage; };
    auto stage_k = [&](int st) { return sRing + st * L::kStage + L::kKV; };
    auto stage_p = [&](int st) { return sRing + st * L::kStage + 2 * L::kKV; };
    auto stage_g = [&](int st) { return sRing + st * L::kStage + 2 * L::kKV + L::kPG; };
    // TMA loads of one step into its stage (thread 0; out-of-range rows and
    // keys arrive as zeros); step 0 also brings the dO tile
    auto issue = [&](int step) {
        if (step >= nsteps) return;
        const int st = step % L::kStages, j0 = step * L::kKeys;
        const uint32_t full = bar_full(st);
        mbar_arrive_expect_tx(full, 2 * L::kKV + (has_g ? 2 : 1) * L::kPG + (step == 0 ? 128 * D * 2 : 0));
        if (step == 0)
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sDO + c * 16384, &tm_go, full, c * 64, pick(ord.go & 3, r0, h, b),
                            pick((ord.go >> 2) & 3, r0, h, b), pick((ord.go >> 4) & 3, r0, h, b));
        for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(stage_v(st) + c * 8192, &tm_v, full, c * 64, pick(ord.v & 3, j0, hk, b),
                        pick((ord.v >> 2) & 3, j0, hk, b), pick((ord.v >> 4) & 3, j0, hk, b));
            tma_load_4d(stage_k(st) + c * 8192, &tm_k, full, c * 64, pick(ord.k & 3, j0, hk, b),
                        pick((ord.k >> 2) & 3, j0, hk, b), pick((ord.k >> 4) & 3, j0, hk, b));
        }
        tma_load_4d(stage_p(st), &tm_p, full, j0, pick(ord.p & 3, r0, h, b), pick((ord.p >> 2) & 3, r0, h, b),
                    pick((ord.p >> 4) & 3, r0, h, b));
        if (has_g)
            tma_load_4d(stage_g(st), &tm_g, full, j0, pick(ord.g & 3, r0, h, b), pick((ord.g >> 2) & 3, r0, h, b),
                        pick((ord.g >> 4) & 3, r0, h, b));
    };
    tc_fence_before();
    __syncthreads();  // barriers initialised
    tc_fence_after();
    if (threadIdx.x == 0) {
        issue(0);
        issue(1);
    }
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc_dp = idesc_f16(128, 64, kBF16, false);
    constexpr uint32_t idesc_pk = idesc_f16(128, D, kBF16, true);
    uint32_t phase_dp = 0, phase_a = 0;
    float r_acc = 0.f;

    for (int step = 0; step < nsteps; ++step) {
        const int st = step % L::kStages;
        const uint32_t sV = stage_v(st), sK = stage_k(st), sP = stage_p(st), sG = stage_g(st);
        wait_bar(bar_full(st), (step / L::kStages) & 1, abort_flag, 8, 3);
        tc_fence_after();
        if (threadIdx.x == 0) {
            // dP = dO V_j^T (N = 64 keys)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                tc_mma_f16(tmem, sw128_desc(sDO + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                           sw128_desc(sV + (kk / 4) * 8192 + (kk % 4) * 32, 16, 1024), idesc_dp, kk > 0 ? 1u : 0u);
            // Bp += P_j K_j (K = 64 keys)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem + tB, sw128_desc(sP + kk * 32, 16, 1024), sw128_desc(sK + kk * 2048, 8192, 1024),
                           idesc_pk, (step > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_dp);
        }
        // the previous step's A products were issued before this step's: once
        // they are done its stage takes the loads two steps ahead
        if (step > 0) {
            wait_bar(bar_a, phase_a, abort_flag, 8, 1);
            phase_a ^= 1u;
        }
        if (threadIdx.x == 0) issue(step + 2);
        wait_bar(bar_dp, phase_dp, abort_flag, 8, 0);
        phase_dp ^= 1u;
        tc_fence_after();
        {
            // this warpgroup's 32 keys (chunks 4 wg .. 4 wg + 3) of row t
            float dp[32];
            tmem_ld32(tmem + lane_base + wg * 32, dp);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t ap = sw_chunk(sP, t, 4 * wg + c), ag = sw_chunk(sG, t, 4 * wg + c);
                uint32_t pw[4], gw[4] = {0u, 0u, 0u, 0u};
                ld_shared_v4(ap, pw);
                if (has_g) ld_shared_v4(ag, gw);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 pp = unpack_pair<T>(pw[e]), gg = unpack_pair<T>(gw[e]);
                    const float e0 = pp.x * (dp[8 * c + 2 * e] + gg.x), e1 = pp.y * (dp[8 * c + 2 * e + 1] + gg.y);
                    acc += e0 + e1;
                    hi[e] = Pack<T>::two(e0, e1);
                    const float2 hh = unpack_pair<T>(hi[e]);
                    lo[e] = Pack<T>::two(e0 - hh.x, e1 - hh.y);
                }
                st_shared_v4(ap, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(ag, lo[0], lo[1], lo[2], lo[3]);
            }
            r_acc += acc;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc_fence_after();
            // A += E_hi K_j + E_lo K_j
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem + tA, sw128_desc(sP + kk * 32, 16, 1024), sw128_desc(sK + kk * 2048, 8192, 1024),
                           idesc_pk, (step > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem + tA, sw128_desc(sG + kk * 32, 16, 1024), sw128_desc(sK + kk * 2048, 8192, 1024),
                           idesc_pk, 1u);
            tc_commit(bar_a);
        }
    }
    wait_bar(bar_a, phase_a, abort_flag, 8, 2);
    tc_fence_after();

    stat[wg * 128 + t] = r_acc;
    __syncthreads();
    const float r = stat[t] + stat[128 + t];
    if (wg == 0 && t < nrows) io.rowsum[((long long)b * io.Hq + h) * io.Sq + r0 + t] = r;

    // dQ = scale (A - r Bp): warpgroup w writes columns [w D/2, (w+1) D/2) of row t
    {
        T* drow = static_cast<T*>(io.dq) + b * io.sdq0 + h * io.sdq1 + (long long)(r0 + t) * io.sdq2 + wg * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            float va[32], vb[32];
            tmem_ld32(tmem + lane_base + tA + wg * (D / 2) + c * 32, va);
            tmem_ld32(tmem + lane_base + tB + wg * (D / 2) + c * 32, vb);
            if (t < nrows) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = io.scale * fmaf(-r, vb[u * 8 + e], va[u * 8 + e]);
                    uint4 pk;
                    pk.x = Pack<T>::two(o[0], o[1]);
                    pk.y = Pack<T>::two(o[2], o[3]);
                    pk.z = Pack<T>::two(o[4], o[5]);
                    pk.w = Pack<T>::two(o[6], o[7]);
                    *reinterpret_cast<uint4*>(drow + c * 32 + u * 8) = pk;
                }
            }
        }
    }
    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (*abort_flag)
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        tmem_dealloc(tmem, kCols);
    }
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Keys kernel layout: V_j once; a two-stage ring of 64-query steps (dO_i, Q_i
// as [64, D] tiles, P_ij and dprobs_ij as [64, 128] tiles, the 64 row sums);
// the dS^T tile [128 keys, 64 queries].
template <int D>
struct BwdKeysSmem {
    static constexpr int kStages = 2;
    static constexpr int kQ = 64;                 // queries per step
    static constexpr int kQD = kQ * D * 2;        // [64, D] tile
    static constexpr int kPG = kQ * 128 * 2;      // [64, 128] tile
    static constexpr int kStage = 2 * kQD + 2 * kPG + 1024;
    static constexpr int kOffV = 0;
    static constexpr int kOffRing = 128 * D * 2;
    static constexpr int kOffS = kOffRing + kStages * kStage;
    static constexpr int kOffBar = kOffS + 128 * kQ * 2;
    static constexpr int kSmem = kOffBar + 64 + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// CTA per 128-key tile of one key/value head; steps over the group's query
// heads and 64-row query tiles.  Per step: dP^T = V_j dO_i^T (lanes = keys),
// dV += P_ij^T dO_i (A read MN-major from the [query][key] tile),
// dS^T = P^T * (dP^T + dprobs^T - r) written row-per-thread as a K-major tile,
// dK += dS^T Q_i.  TMEM: dP^T [0, 64), dV [64, 64 + D), dK [64 + D, 64 + 2D).
template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_tc_keys_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_go,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_p,
                   const __grid_constant__ CUtensorMap tm_g, const BwdIO io, const BwdOrd ord) {
    using L = BwdKeysSmem<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kCols = 64 + 2 * D <= 256 ? 256 : 512;
    constexpr uint32_t tDV = 64, tDK = 64 + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sV = smem_u32(smem + L::kOffV), sRing = smem_u32(smem + L::kOffRing);
    const uint32_t sS = smem_u32(smem + L::kOffS);
    // [0] dP^T and dV done, [1] dK done, [2 + stage] stage loaded
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 + L::kStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, wg = threadIdx.x / 128, t = threadIdx.x % 128;
    const int kt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int j0 = kt * 128, ncols = min(128, io.Skv - j0);
    const int nq = (io.Sq + L::kQ - 1) / L::kQ;
    const int nsteps = io.group * nq;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t bar_dp = smem_u32(&bars[0]), bar_k = smem_u32(&bars[1]);

    auto bar_full = [&](int st) { return smem_u32(&bars[2 + st]); };
    const bool has_g = io.gp != nullptr;
    if (threadIdx.x == 0) {
        mbar_init(bar_dp, 1);
        mbar_init(bar_k, 1);
        for (int st = 0; st < L::kStages; ++st) mbar_init(bar_full(st), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_go);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_p);
        if (has_g) prefetch_tmap(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kCols);
        tmem_relinquish();
    }
    auto st_do = [&](int st) { return sRing + st * L::kStage; };
    auto st_q = [&](int st) { return sRing + st * L::kStage + L::kQD; };
    auto st_p = [&](int st) { return sRing + st * L::kStage + 2 * L::kQD; };
    auto st_g = [&](int st) { return sRing + st * L::kStage + 2 * L::kQD + L::kPG; };
    auto st_r = [&](int st) { return sRing + st * L::kStage + 2 * L::kQD + 2 * L::kPG; };
    // TMA loads of one step into its stage (thread 0; out-of-range rows and
    // keys arrive as zeros); step 0 also brings the V tile
    auto issue_tma = [&](int step) {
        if (step >= nsteps) return;
        const int st = step % L::kStages;
        const int h = hk * io.group + step / nq, r0 = (step % nq) * L::kQ;
        const uint32_t full = bar_full(st);
        mbar_arrive_expect_tx(full, 2 * L::kQD + (has_g ? 2 : 1) * L::kPG + (step == 0 ? 128 * D * 2 : 0));
        if (step == 0)
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sV + c * 16384, &tm_v, full, c * 64, pick(ord.v & 3, j0, hk, b),
                            pick((ord.v >> 2) & 3, j0, hk, b), pick((ord.v >> 4) & 3, j0, hk, b));
        for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(st_do(st) + c * 8192, &tm_go, full, c * 64, pick(ord.go & 3, r0, h, b),
                        pick((ord.go >> 2) & 3, r0, h, b), pick((ord.go >> 4) & 3, r0, h, b));
            tma_load_4d(st_q(st) + c * 8192, &tm_q, full, c * 64, pick(ord.q & 3, r0, h, b),
                        pick((ord.q >> 2) & 3, r0, h, b), pick((ord.q >> 4) & 3, r0, h, b));
        }
        for (int c = 0; c < 2; ++c) {  // the two 64-key halves
            tma_load_4d(st_p(st) + c * 8192, &tm_p, full, j0 + 64 * c, pick(ord.p & 3, r0, h, b),
                        pick((ord.p >> 2) & 3, r0, h, b), pick((ord.p >> 4) & 3, r0, h, b));
            if (has_g)
                tma_load_4d(st_g(st) + c * 8192, &tm_g, full, j0 + 64 * c, pick(ord.g & 3, r0, h, b),
                            pick((ord.g >> 2) & 3, r0, h, b), pick((ord.g >> 4) & 3, r0, h, b));
        }
    };
    // row sums of a step's queries: 4-byte copies, one commit group per step
    auto issue_r = [&](int step) {
        if (step < nsteps && threadIdx.x < L::kQ) {
            const int st = step % L::kStages;
            const int h = hk * io.group + step / nq, r0 = (step % nq) * L::kQ, nrows = min(L::kQ, io.Sq - r0);
            const bool ok = (int)threadIdx.x < nrows;
            const float* src = io.rowsum + ((long long)b * io.Hq + h) * io.Sq + r0 + (ok ? threadIdx.x : 0);
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(st_r(st) + 4 * threadIdx.x), "l"(src),
                         "r"(ok ? 4 : 0)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    tc_fence_before();
    __syncthreads();  // barriers initialised
    tc_fence_after();
    if (threadIdx.x == 0) issue_tma(0);
    issue_r(0);
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc_dpt = idesc_f16(128, L::kQ, kBF16, false);
    constexpr uint32_t idesc_dv = idesc_f16(128, D, kBF16, true) | (1u << 15);  // A MN-major too
    constexpr uint32_t idesc_dk = idesc_f16(128, D, kBF16, true);
    uint32_t phase_dp = 0, phase_k = 0;
    const int key = t;  // this thread's TMEM lane and row of the dS^T tile

    for (int step = 0; step < nsteps; ++step) {
        const int st = step % L::kStages;
        const uint32_t sDO = st_do(st), sQ = st_q(st), sP = st_p(st), sG = st_g(st);
        const float* rs = reinterpret_cast<const float*>(smem + (st_r(st) - smem_u32(smem)));
        asm volatile("cp.async.wait_group 0;" ::: "memory");  // this step's row sums
        wait_bar(bar_full(st), (step / L::kStages) & 1, abort_flag, 9, 3);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (threadIdx.x == 0) {
            // dP^T = V_j dO_i^T (M = 128 keys, N = 64 queries, K = D)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                tc_mma_f16(tmem, sw128_desc(sV + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024),
                           sw128_desc(sDO + (kk / 4) * 8192 + (kk % 4) * 32, 16, 1024), idesc_dpt, kk > 0 ? 1u : 0u);
            // dV += P^T dO_i (M = 128 keys, N = D, K = 64 queries; both operands MN-major)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem + tDV, sw128_desc(sP + kk * 2048, 8192, 1024), sw128_desc(sDO + kk * 2048, 8192, 1024),
                           idesc_dv, (step > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_dp);
        }
        // dK of the previous step (issued before this step's products) frees
        // the other stage and the dS^T tile
        if (step > 0) {
            wait_bar(bar_k, phase_k, abort_flag, 9, 1);
            phase_k ^= 1u;
        }
        if (threadIdx.x == 0) issue_tma(step + 1);
        issue_r(step + 1);
        wait_bar(bar_dp, phase_dp, abort_flag, 9, 0);
        phase_dp ^= 1u;
        tc_fence_after();
        {
            // queries [32 wg, 32 wg + 32) of key `key`
            float dpt[32];
            tmem_ld32(tmem + lane_base + wg * 32, dpt);
            const uint32_t kcol = (key >> 6) * 8192 + (key & 7) * 2;
            const uint32_t kchunk = (key & 63) >> 3;
            uint32_t out[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float ds[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int q = wg * 32 + e + u;
                    const uint32_t off = kcol + q * 128 + ((kchunk ^ (q & 7)) << 4);
                    const float pv = Pack<T>::load_bits(lds_u16(sP + off));
                    const float gv = has_g ? Pack<T>::load_bits(lds_u16(sG + off)) : 0.f;
                    ds[u] = pv * (dpt[e + u] + gv - rs[q]);
                }
                out[e / 2] = Pack<T>::two(ds[0], ds[1]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                st_shared_v4(sS + key * 128 + (((4 * wg + c) ^ (key & 7)) << 4), out[4 * c], out[4 * c + 1],
                             out[4 * c + 2], out[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x == 0) {
            tc_fence_after();
            // dK += dS^T Q_i (M = 128 keys, N = D, K = 64 queries)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem + tDK, sw128_desc(sS + kk * 32, 16, 1024), sw128_desc(sQ + kk * 2048, 8192, 1024),
                           idesc_dk, (step > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar_k);
        }
    }
    wait_bar(bar_k, phase_k, abort_flag, 9, 2);
    tc_fence_after();

    // dV (warpgroup 0) and dK (warpgroup 1) rows: lane t is key j0 + t
    {
        const bool is_k = wg == 1;
        T* drow = is_k ? static_cast<T*>(io.dk) + b * io.sdk0 + hk * io.sdk1 + (long long)(j0 + t) * io.sdk2
                       : static_cast<T*>(io.dv) + b * io.sdv0 + hk * io.sdv1 + (long long)(j0 + t) * io.sdv2;
        const float sc = is_k ? io.scale : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float v[32];
            tmem_ld32(tmem + lane_base + (is_k ? tDK : tDV) + c * 32, v);
            if (t < ncols) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    uint4 pk;
                    pk.x = Pack<T>::two(sc * v[u * 8 + 0], sc * v[u * 8 + 1]);
                    pk.y = Pack<T>::two(sc * v[u * 8 + 2], sc * v[u * 8 + 3]);
                    pk.z = Pack<T>::two(sc * v[u * 8 + 4], sc * v[u * 8 + 5]);
                    pk.w = Pack<T>::two(sc * v[u * 8 + 6], sc * v[u * 8 + 7]);
                    *reinterpret_cast<uint4*>(drow + c * 32 + u * 8) = pk;
                }
            }
        }
    }
    __syncwarp();  // each warp reaches the CTA-wide barrier converged: lane-0 roles end later than their warp
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        if (*abort_flag)
            for (int i = 0; i < 200; ++i) __nanosleep(1000);
        tmem_dealloc(tmem, kCols);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 4-D tensor map over a logical [B, H, S, X] tensor (X contiguous) with a box
// of 64 x box_rows rows, 128-byte swizzle.  The three outer dims are ordered by
// stride; `ord` receives the packed order code.
bool encode_map(CUtensorMap* map, int dtype, const void* base, long long X, long long S, long long H, long long Bn,
                const int64_t* st /* [B, H, S] element strides */, uint32_t box_rows, uint32_t* ord) {
    auto fn = encode_fn();
    if (!fn) return false;
    struct Dim { long long ext, stride; int sel; };
    Dim d[3] = {{S, st[2], 1}, {H, st[1], 2}, {Bn, st[0], 3}};
    // a broadcast dimension (stride 0, every index reads the same memory)
    // becomes an extent-1 dimension whose coordinate is always 0 (code 0)
    for (auto& x : d)
        if (x.ext > 1 && x.stride == 0) { x.ext = 1; x.sel = 0; }
    // extent-1 dims never move: give them a stride past everything else,
    // rounded up to the 16 bytes every tensor-map stride needs (a single P
    // row of 698 keys, say, is still a valid map)
    long long maxb = X;
    for (auto& x : d) if (x.ext > 1) maxb = std::max(maxb, x.stride * x.ext);
    maxb = (maxb + 7) / 8 * 8;
    for (auto& x : d) if (x.ext <= 1) x.stride = maxb;
    std::stable_sort(d, d + 3, [](const Dim& a, const Dim& c) { return a.stride < c.stride; });
    cuuint64_t dims[4] = {(cuuint64_t)X, 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {64, 1, 1, 1};
    uint32_t code = 0;
    for (int k = 0; k < 3; ++k) {
        dims[k + 1] = (cuuint64_t)d[k].ext;
        strides[k] = (cuuint64_t)(d[k].stride * 2);
        if (strides[k] % 16 != 0) return false;
        box[k + 1] = d[k].sel == 1 ? box_rows : 1;
        code |= (uint32_t)d[k].sel << (2 * k);
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *ord = code;
    return r == CUDA_SUCCESS;
}

// Small cache of encoded tensor maps, so that repeated calls on the same
// buffers skip the host-side encode.  Keyed by everything the encode reads.
struct MapKey {
    const void* base;
    long long X, S, H, Bn, s0, s1, s2;
    int dtype;
    uint32_t box_rows;
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    uint32_t ord;
    bool used;
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool make_map(CUtensorMap* map, int dtype, const void* base, long long X, long long S, long long H, long long Bn,
              const int64_t* st, uint32_t box_rows, uint32_t* ord) {
    MapKey key;
    std::memset(&key, 0, sizeof(key));
    key.base = base; key.X = X; key.S = S; key.H = H; key.Bn = Bn;
    key.s0 = st[0]; key.s1 = st[1]; key.s2 = st[2]; key.dtype = dtype; key.box_rows = box_rows;
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (auto& e : g_maps)
        if (e.used && e.key == key) {
            *map = e.map;
            *ord = e.ord;
            return true;
        }
    if (!encode_map(map, dtype, base, X, S, H, Bn, st, box_rows, ord)) return false;
    MapEntry& e = g_maps[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCache;
    e.key = key;
    e.map = *map;
    e.ord = *ord;
    e.used = true;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool strides_ok(const int64_t* st, const int64_t* ext) {
    for (int i = 0; i < 3; ++i)
        if (ext[i] > 1 && st[i] % 8 != 0) return false;
    return true;
}

// A tensor whose rows are broadcast (row stride 0 over more than one row)
// cannot be read as 128-row TMA boxes; batch and head broadcasts can (see
// encode_map).
bool rows_broadcast(const int64_t* st, int64_t rows) { return rows > 1 && st[2] == 0; }

// One-time (per kernel instantiation and device) launch preparation: the
// register check of the in-kernel split and the shared-memory opt-in.  Keyed
// by the kernel's address (every instantiation has the same pointer type).
struct Prepared {
    const void* kern;
    int dev;
    int state;  // 1 = ready, 2 = refused
};
std::mutex g_prep_mu;
Prepared g_prep[64];
int g_prep_n = 0;

template <typename K>
cudaError_t prepare_kernel(K kern, int smem, bool reg_split = true) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void* key = reinterpret_cast<const void*>(kern);
    std::lock_guard<std::mutex> lock(g_prep_mu);
    for (int i = 0; i < g_prep_n; ++i)
        if (g_prep[i].kern == key && g_prep[i].dev == dev)
            return g_prep[i].state == 1 ? cudaSuccess : cudaErrorNotSupported;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    int state = 1;
    // the in-kernel register split must fit what the launch allocates
    if (reg_split && fa.numRegs * kThreads < (int)(128 * kRegsLow + 256 * kRegsHigh)) state = 2;
    if (state == 1) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    if (g_prep_n < 64) g_prep[g_prep_n++] = Prepared{key, dev, state};
    return state == 1 ? cudaSuccess : cudaErrorNotSupported;
}

template <int D, typename T, bool kMasked, int QT>
cudaError_t launch_twopass(const Problem& p, cudaStream_t stream) {
    using C = TcCfg<D, QT>;
    CUtensorMap mq, mk, mv, mp, mo;
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    if (!make_map(&mq, p.dtype, p.q, p.D, p.Sq, p.Hq, p.B, p.sq, 128, &prm.ord_q) ||
        !make_map(&mk, p.dtype, p.k, p.D, p.Skv, p.Hkv, p.B, p.sk, 128, &prm.ord_k) ||
        !make_map(&mv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, 128, &prm.ord_v) ||
        !make_map(&mp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, 32, &prm.ord_p) ||
        !make_map(&mo, p.dtype, p.o, p.Dv, p.Sq, p.Hq, p.B, p.so, 32, &prm.ord_o))
        return cudaErrorNotSupported;
    prm.Sq = (int)p.Sq;
    prm.Skv = (int)p.Skv;
    prm.Hq = (int)p.Hq;
    prm.group = (int)p.group;
    prm.n_qtiles = (int)((p.Sq + 127) / 128);
    prm.causal = p.causal;
    prm.c2 = p.scale * kLog2e;
    prm.mask = p.mask;
    prm.mask_kind = p.mask_kind;
    prm.mask_dtype = p.mask_dtype;
    prm.sm0 = p.sm[0]; prm.sm1 = p.sm[1]; prm.sm2 = p.sm[2];
    prm.o = p.o;
    prm.so0 = p.so[0]; prm.so1 = p.so[1]; prm.so2 = p.so[2];
    prm.lse = p.lse;
    prm.p = p.p;
    prm.sp0 = p.sp[0]; prm.sp1 = p.sp[1]; prm.sp2 = p.sp[2];
    auto kern = tc_twopass_kernel<D, T, kMasked, QT>;
    cudaError_t e = prepare_kernel(kern, C::kSmem);
    if (e != cudaSuccess) return e;
    const unsigned nz = QT == 2 ? (unsigned)((prm.n_qtiles + 1) / 2) : (unsigned)prm.n_qtiles;
    dim3 grid((unsigned)p.Hq, (unsigned)p.B, nz);
    kern<<<grid, kThreads, C::kSmem, stream>>>(mq, mk, mv, mp, mo, prm);
    return cudaGetLastError();
}

template <int D, typename T, bool kMasked>
cudaError_t launch_wide(const Problem& p, cudaStream_t stream) {
    using C = WideCfg<D>;
    CUtensorMap mq, mk, mv, mp, mo;
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    if (!make_map(&mq, p.dtype, p.q, p.D, p.Sq, p.Hq, p.B, p.sq, 128, &prm.ord_q) ||
        !make_map(&mk, p.dtype, p.k, p.D, p.Skv, p.Hkv, p.B, p.sk, 128, &prm.ord_k) ||
        !make_map(&mv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, 128, &prm.ord_v) ||
        !make_map(&mp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, 32, &prm.ord_p) ||
        !make_map(&mo, p.dtype, p.o, p.Dv, p.Sq, p.Hq, p.B, p.so, 32, &prm.ord_o))
        return cudaErrorNotSupported;
    prm.Sq = (int)p.Sq;
    prm.Skv = (int)p.Skv;
    prm.Hq = (int)p.Hq;
    prm.group = (int)p.group;
    prm.n_qtiles = (int)((p.Sq + 127) / 128);
    prm.causal = p.causal;
    prm.c2 = p.scale * kLog2e;
    prm.mask = p.mask;
    prm.mask_kind = p.mask_kind;
    prm.mask_dtype = p.mask_dtype;
    prm.sm0 = p.sm[0]; prm.sm1 = p.sm[1]; prm.sm2 = p.sm[2];
    prm.o = p.o;
    prm.so0 = p.so[0]; prm.so1 = p.so[1]; prm.so2 = p.so[2];
    prm.lse = p.lse;
    prm.p = p.p;
    prm.sp0 = p.sp[0]; prm.sp1 = p.sp[1]; prm.sp2 = p.sp[2];
    auto kern = tc_wide_kernel<D, T, kMasked>;
    cudaError_t e = prepare_kernel(kern, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.Hq, (unsigned)p.B, (unsigned)prm.n_qtiles);
    kern<<<grid, kThreads, C::kSmem, stream>>>(mq, mk, mv, mp, mo, prm);
    return cudaGetLastError();
}

int sm_count();  // SMs of the current device (cached)

template <int D, typename T, bool kMasked>
cudaError_t launch_fused(const Problem& p, cudaStream_t stream) {
    using L = FusedSmem<D>;
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.Sq = (int)p.Sq;
    prm.Skv = (int)p.Skv;
    prm.Hq = (int)p.Hq;
    prm.group = (int)p.group;
    prm.n_qtiles = (int)((p.Sq + 127) / 128);
    prm.causal = p.causal;
    prm.c2 = p.scale * kLog2e;
    prm.mask = p.mask;
    prm.mask_kind = p.mask_kind;
    prm.mask_dtype = p.mask_dtype;
    prm.sm0 = p.sm[0]; prm.sm1 = p.sm[1]; prm.sm2 = p.sm[2];
    prm.o = p.o;
    prm.so0 = p.so[0]; prm.so1 = p.so[1]; prm.so2 = p.so[2];
    prm.lse = p.lse;
    prm.p = p.p;
    prm.sp0 = p.sp[0]; prm.sp1 = p.sp[1]; prm.sp2 = p.sp[2];
    FusedIO io;
    std::memset(&io, 0, sizeof(io));
    io.q = p.q; io.sq0 = p.sq[0]; io.sq1 = p.sq[1]; io.sq2 = p.sq[2];
    io.k = p.k; io.sk0 = p.sk[0]; io.sk1 = p.sk[1]; io.sk2 = p.sk[2];
    io.v = p.v; io.sv0 = p.sv[0]; io.sv1 = p.sv[1]; io.sv2 = p.sv[2];
    const uint32_t need = (uint32_t)(max_live_key_tiles(p.Sq, p.Skv, p.causal != 0) * 128 + D);
    io.tmem_cols = need <= 256 ? 256u : 512u;
    // a grid that leaves most SMs idle takes 32-row query groups instead of
    // 128-row tiles (four times the CTAs, each a quarter of the rows to
    // finish and copy out), as long as the finer grid still fits one wave
    io.rpc = p.B * p.Hq * prm.n_qtiles * 4 <= sm_count() ? 32 : 128;
    auto kern = tc_fused_kernel<D, T, kMasked>;
    cudaError_t e = prepare_kernel(kern, L::kSmem, false);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.Hq, (unsigned)p.B, (unsigned)((p.Sq + io.rpc - 1) / io.rpc));
    kern<<<grid, FusedCfg::kThreads, L::kSmem, stream>>>(prm, io);
    return cudaGetLastError();
}

// Clusters of `cl` CTAs of the one-sweep kernel that can be resident at once
// on this device (0 when none can be placed), cached per (kernel, size).
struct ClusterFit {
    const void* kern;
    int dev, cl, n;
};
std::mutex g_fit_mu;
ClusterFit g_fit[32];
int g_fit_n = 0;

template <typename K>
int resident_clusters(K kern, int cl, int smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const void* key = reinterpret_cast<const void*>(kern);
    std::lock_guard<std::mutex> lock(g_fit_mu);
    for (int i = 0; i < g_fit_n; ++i)
        if (g_fit[i].kern == key && g_fit[i].dev == dev && g_fit[i].cl == cl) return g_fit[i].n;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)cl, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (g_fit_n < 32) g_fit[g_fit_n++] = ClusterFit{key, dev, cl, n};
    return n;
}

// CTAs per cluster of the one-sweep kernel: enough that no CTA keeps more
// than kMaxOwn key tiles of a query block (0: the rows are too long).
int onesweep_cluster(const Problem& p) {
    const int64_t n = max_live_key_tiles(p.Sq, p.Skv, p.causal != 0);
    const int64_t cl = (n + 3) / 4;
    return cl >= 1 && cl <= kOneMaxCluster ? (int)cl : 0;
}

template <int D, typename T, bool kMasked>
cudaError_t launch_onesweep(const Problem& p, cudaStream_t stream) {
    using C = OneCfg<D>;
    static_assert(C::kMaxOwn == 4, "onesweep_cluster assumes four tiles per CTA");
    const int cl = onesweep_cluster(p);
    if (cl == 0) return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv, mp, mo;
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    // (the O map only validates the layout: O rows are stored with 16-byte stores)
    if (!make_map(&mq, p.dtype, p.q, p.D, p.Sq, p.Hq, p.B, p.sq, 128, &prm.ord_q) ||
        !make_map(&mk, p.dtype, p.k, p.D, p.Skv, p.Hkv, p.B, p.sk, 128, &prm.ord_k) ||
        !make_map(&mv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, 128, &prm.ord_v) ||
        !make_map(&mp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, 32, &prm.ord_p) ||
        !make_map(&mo, p.dtype, p.o, p.Dv, p.Sq, p.Hq, p.B, p.so, 32, &prm.ord_o))
        return cudaErrorNotSupported;
    prm.Sq = (int)p.Sq;
    prm.Skv = (int)p.Skv;
    prm.Hq = (int)p.Hq;
    prm.group = (int)p.group;
    prm.n_qtiles = (int)((p.Sq + 127) / 128);
    prm.causal = p.causal;
    prm.B = (int)p.B;
    prm.cl = cl;
    prm.c2 = p.scale * kLog2e;
    prm.mask = p.mask;
    prm.mask_kind = p.mask_kind;
    prm.mask_dtype = p.mask_dtype;
    prm.sm0 = p.sm[0]; prm.sm1 = p.sm[1]; prm.sm2 = p.sm[2];
    prm.o = p.o;
    prm.so0 = p.so[0]; prm.so1 = p.so[1]; prm.so2 = p.so[2];
    prm.lse = p.lse;
    prm.p = p.p;
    prm.sp0 = p.sp[0]; prm.sp1 = p.sp[1]; prm.sp2 = p.sp[2];
    auto kern = tc_onesweep_kernel<D, T, kMasked>;
    cudaError_t e = prepare_kernel(kern, C::kSmem);
    if (e != cudaSuccess) return e;
    const int fit = resident_clusters(kern, cl, C::kSmem);
    if (fit <= 0) return cudaErrorNotSupported;
    const long long items = p.B * p.Hq * (long long)prm.n_qtiles;
    if (items > (1ll << 30)) return cudaErrorNotSupported;
    int G = (int)(items < fit ? items : fit);
    // test / profiling hook: fewer clusters, so each walks more query blocks
    const char* cap_env = std::getenv("SDPA_MATH_ONESWEEP_CLUSTERS");
    const int cap = cap_env ? std::atoi(cap_env) : 0;
    if (cap > 0 && cap < G) G = cap;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(G * cl), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)C::kSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mp, prm);
    return e;
}

int sm_count() {
    static int n = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return 148;
        return v;
    }();
    return n;
}

}  // namespace

// Query tiles per CTA: two tiles share every K / V load (half the load traffic
// per score tile) when that still gives about three quarters of a CTA per SM.
// Measured on GB300 (96 shapes, D 64 / 128): the paired layout wins from about
// 0.75 pairs per SM, with or without a causal mask, except where a paired
// CTA's two unequal causal streams cost more than the shared loads save:
// causal calls past two pairs per SM (1-2 % slower at 512 pairs) and causal
// D = 128 rows of more than 8 key tiles (2k: 47.1 against 45.8 us).
int tc_query_tiles(const Problem& p) {
    const int64_t nq = (p.Sq + 127) / 128;
    if (nq < 2) return 1;
    const int64_t pairs = p.B * p.Hq * ((nq + 1) / 2);
    const int64_t sms = sm_count();
    if (pairs * 4 < sms * 3) return 1;
    if (p.causal && (pairs > 2 * sms || (p.D > 64 && nq > 8))) return 1;
    return 2;
}

// Whether AUTO takes the one-sweep cluster kernel: causal calls whose row
// blocks need clusters of two or more CTAs and whose clusters all fit in one
// wave (row blocks x cluster size <= SMs).  There its shorter per-block
// critical path wins (1x8x8 1024x1024 causal: 16.1 against 20.5 us at D = 64,
// 18.1 against 22.1 us at D = 128); everywhere else on the same sweep it lost.
bool onesweep_auto(const Problem& p) {
    if (!p.causal) return false;
    const int64_t n = max_live_key_tiles(p.Sq, p.Skv, true);
    const int64_t cl = (n + 3) / 4;
    if (cl < 2 || cl > 8) return false;
    const int64_t blocks = p.B * p.Hq * ((p.Sq + 127) / 128);
    return blocks * cl <= (int64_t)sm_count();
}

namespace {

template <typename T, int QT>
cudaError_t launch_qt(const Problem& p, cudaStream_t stream) {
    const bool masked = p.mask_kind != kMaskNone;
    if constexpr (QT == 1) {
        if (p.D == 64) return masked ? launch_wide<64, T, true>(p, stream) : launch_wide<64, T, false>(p, stream);
        return masked ? launch_wide<128, T, true>(p, stream) : launch_wide<128, T, false>(p, stream);
    }
    if (p.D == 64)
        return masked ? launch_twopass<64, T, true, QT>(p, stream) : launch_twopass<64, T, false, QT>(p, stream);
    return masked ? launch_twopass<128, T, true, QT>(p, stream) : launch_twopass<128, T, false, QT>(p, stream);
}

template <typename T>
cudaError_t launch_t(const Problem& p, int mode, cudaStream_t stream) {
    if (mode == 4) {
        const bool masked = p.mask_kind != kMaskNone;
        if (p.D == 64) return masked ? launch_onesweep<64, T, true>(p, stream) : launch_onesweep<64, T, false>(p, stream);
        return masked ? launch_onesweep<128, T, true>(p, stream) : launch_onesweep<128, T, false>(p, stream);
    }
    if (mode == 3) {
        const bool masked = p.mask_kind != kMaskNone;
        if (p.D == 64) return masked ? launch_fused<64, T, true>(p, stream) : launch_fused<64, T, false>(p, stream);
        return masked ? launch_fused<128, T, true>(p, stream) : launch_fused<128, T, false>(p, stream);
    }
    return mode == 2 ? launch_qt<T, 2>(p, stream) : launch_qt<T, 1>(p, stream);
}

}  // namespace

bool tc_supports(const Problem& p, bool fused, const char** why) {
    if (p.dtype != kF16 && p.dtype != kBF16) { *why = "dtype must be f16 or bf16"; return false; }
    if (p.D != p.Dv || (p.D != 64 && p.D != 128)) { *why = "head dim must be 64 or 128 (D == Dv)"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (!(p.scale > 0.f)) { *why = "scale must be positive"; return false; }
    if (p.Sq >= (1ll << 31) || p.Skv >= (1ll << 31) || p.B > 65535 || p.Sq > 65535ll * 128) {
        *why = "sizes beyond the grid limits"; return false;
    }
    const int64_t eq[3] = {p.B, p.Hq, p.Sq}, ek[3] = {p.B, p.Hkv, p.Skv};
    if (fused) {
        // plain 16-byte loads of q / k / v rows and stores of O rows; P rows
        // may have any alignment
        if (max_live_key_tiles(p.Sq, p.Skv, p.causal != 0) > 2) {
            *why = "the fused kernel keeps at most two live 128-key tiles per row block in TMEM"; return false;
        }
        if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.o)) {
            *why = "q, k, v and out must be 16-byte aligned"; return false;
        }
        if (!strides_ok(p.sq, eq) || !strides_ok(p.sk, ek) || !strides_ok(p.sv, ek) || !strides_ok(p.so, eq)) {
            *why = "q, k, v and out rows must start on 16-byte boundaries"; return false;
        }
        return true;
    }
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.p) || !aligned16(p.o)) {
        *why = "q, k, v, out and probs must be 16-byte aligned"; return false;
    }
    if (!strides_ok(p.sq, eq) || !strides_ok(p.sk, ek) || !strides_ok(p.sv, ek) || !strides_ok(p.sp, eq) ||
        !strides_ok(p.so, eq)) {
        *why = "outer strides must be multiples of 8 elements (16 bytes)"; return false;
    }
    if (rows_broadcast(p.sq, p.Sq) || rows_broadcast(p.sk, p.Skv) || rows_broadcast(p.sv, p.Skv)) {
        *why = "q, k or v rows are broadcast (row stride 0): TMA tiles need distinct rows"; return false;
    }
    return true;
}

// ---- tensor-core decode / split-KV (host)
namespace {
// Cluster size, key chunk, ring stages and shared-memory layout of
// tc_decode_kernel for C CTAs per cluster; false when it does not fit.
bool plan_tc_decode(const Problem& p, int C, TcDecParams* dp, int* smem) {
    const long long rows = p.group * p.Sq;
    const long long chunk = (p.Skv + C - 1) / C;
    // two stages keep a CTA near 110 KB (with 4 rows and 2048-key chunks), so
    // two CTAs share an SM and cover each other's load latency
    const int stages = 2;
    const long long shrink = stages == 2 ? DecLayout::kRingShrink2 : 0;
    long long off = DecLayout::kFixed - shrink;
    auto al = [](long long x) { return (x + 15) & ~15ll; };
    const long long off_ss = off; off = al(off + rows * chunk * 4);
    const long long off_part = off; off = al(off + rows * 128 * 4);
    const long long off_st = off; off += rows * 2 * 4;
    off += 1024;  // alignment slack of the dynamic base
    if (off > kDecSmemMax) return false;
    dp->chunk = (int)chunk;
    dp->stages = stages;
    dp->off_ss = (int)off_ss;
    dp->off_part = (int)off_part;
    dp->off_st = (int)off_st;
    *smem = (int)off;
    return true;
}

int tc_decode_cluster(const Problem& p) {
    const long long c = (p.Skv + 255) / 256;
    return (int)(c < 1 ? 1 : (c > kDecMaxCluster ? kDecMaxCluster : c));
}

std::mutex g_dec_mu;
struct DecChoice { const void* kern; int dev; int smem; int C; };
DecChoice g_dec[32];
int g_ndec = 0;

template <typename T>
cudaError_t launch_tc_decode_t(const Problem& pr, cudaStream_t stream) {
    TcDecParams p;
    std::memset(&p, 0, sizeof(p));
    CUtensorMap mk, mv;
    if (!make_map(&mk, pr.dtype, pr.k, pr.D, pr.Skv, pr.Hkv, pr.B, pr.sk, 128, &p.ord_k) ||
        !make_map(&mv, pr.dtype, pr.v, pr.Dv, pr.Skv, pr.Hkv, pr.B, pr.sv, 128, &p.ord_v))
        return cudaErrorNotSupported;
    p.q = pr.q; p.sq0 = pr.sq[0]; p.sq1 = pr.sq[1]; p.sq2 = pr.sq[2];
    p.mask = pr.mask; p.mask_kind = pr.mask_kind; p.mask_dtype = pr.mask_dtype;
    p.sm0 = pr.sm[0]; p.sm1 = pr.sm[1]; p.sm2 = pr.sm[2];
    p.o = pr.o; p.so0 = pr.so[0]; p.so1 = pr.so[1]; p.so2 = pr.so[2];
    p.p = pr.p; p.sp0 = pr.sp[0]; p.sp1 = pr.sp[1]; p.sp2 = pr.sp[2];
    p.lse = pr.lse;
    p.Hq = (int)pr.Hq; p.Sq = (int)pr.Sq; p.Skv = (int)pr.Skv; p.group = (int)pr.group;
    p.rows = (int)(pr.group * pr.Sq); p.causal = pr.causal;
    p.c2 = pr.scale * kLog2e;
    auto kern = tc_decode_kernel<T>;
    int C = tc_decode_cluster(pr), smem = 0;
    if (!plan_tc_decode(pr, C, &p, &smem)) return cudaErrorNotSupported;
    cudaError_t e = prepare_kernel(kern, kDecSmemMax, false);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (C > 8) {
        // a cluster above the portable size needs the opt-in and a schedulable placement
        std::lock_guard<std::mutex> lock(g_dec_mu);
        int chosen = 0;
        for (int i = 0; i < g_ndec; ++i)
            if (g_dec[i].kern == reinterpret_cast<const void*>(kern) && g_dec[i].dev == dev && g_dec[i].smem == smem)
                chosen = g_dec[i].C;
        if (chosen == 0) {
            int nc = 0;
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
                cfg.gridDim = dim3((unsigned)C, 1, 1);
                cfg.dynamicSmemBytes = (size_t)smem;
                attr[0].val.clusterDim.x = (unsigned)C;
                if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) nc = 0;
            }
            (void)cudaGetLastError();
            chosen = nc > 0 ? C : 8;
            if (g_ndec < 32) g_dec[g_ndec++] = DecChoice{reinterpret_cast<const void*>(kern), dev, smem, chosen};
        }
        if (chosen != C) {
            C = chosen;
            if (!plan_tc_decode(pr, C, &p, &smem)) return cudaErrorNotSupported;
        }
    }
    cfg.gridDim = dim3((unsigned)C, (unsigned)pr.Hkv, (unsigned)pr.B);
    cfg.dynamicSmemBytes = (size_t)smem;
    attr[0].val.clusterDim.x = (unsigned)C;
    e = cudaLaunchKernelEx(&cfg, kern, mk, mv, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

bool tc_decode_supports(const Problem& p, const char** why) {
    if (p.dtype != kF16 && p.dtype != kBF16) { *why = "dtype must be f16 or bf16"; return false; }
    if (p.D != 128 || p.Dv != 128) { *why = "head dims must be 128"; return false; }
    if (p.group * p.Sq > 16) { *why = "more than 16 query rows per key/value head"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (p.B > 65535 || p.Hkv > 65535 || p.Skv >= (1ll << 31)) { *why = "sizes beyond the grid limits"; return false; }
    const int64_t eq[3] = {p.B, p.Hq, p.Sq}, ek[3] = {p.B, p.Hkv, p.Skv};
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !strides_ok(p.sq, eq) || !strides_ok(p.sk, ek) ||
        !strides_ok(p.sv, ek)) {
        *why = "q, k and v rows must start on 16-byte boundaries"; return false;
    }
    if (rows_broadcast(p.sk, p.Skv) || rows_broadcast(p.sv, p.Skv)) {
        *why = "k or v rows are broadcast (row stride 0): TMA tiles need distinct rows"; return false;
    }
    TcDecParams dp;
    int smem;
    if (!plan_tc_decode(p, tc_decode_cluster(p), &dp, &smem)) {
        *why = "the scores of a key chunk do not fit shared memory"; return false;
    }
    return true;
}

cudaError_t launch_tc_decode(const Problem& p, cudaStream_t stream) {
    const char* why;
    if (!tc_decode_supports(p, &why)) return cudaErrorNotSupported;
    return p.dtype == kF16 ? launch_tc_decode_t<__half>(p, stream) : launch_tc_decode_t<__nv_bfloat16>(p, stream);
}

bool bwd_tc_supports(const BwdProblem& p, const char** why) {
    if (p.dtype != kF16 && p.dtype != kBF16) { *why = "dtype must be f16 or bf16"; return false; }
    if (p.D != p.Dv || (p.D != 64 && p.D != 128)) { *why = "head dim must be 64 or 128 (D == Dv)"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (p.Sq >= (1ll << 31) || p.Skv >= (1ll << 31) || p.B > 65535 || p.Hq > 65535) {
        *why = "sizes beyond the grid limits"; return false;
    }
    const void* ptrs[9] = {p.q, p.k, p.v, p.p, p.dout, p.dprobs, p.dq, p.dk, p.dv};
    for (const void* x : ptrs)
        if (x && !aligned16(x)) { *why = "every tensor must be 16-byte aligned"; return false; }
    const int64_t eq[3] = {p.B, p.Hq, p.Sq}, ek[3] = {p.B, p.Hkv, p.Skv};
    if (!strides_ok(p.sq, eq) || !strides_ok(p.sk, ek) || !strides_ok(p.sv, ek) || !strides_ok(p.sp, eq) ||
        !strides_ok(p.sgo, eq) || (p.dprobs && !strides_ok(p.sgp, eq)) || !strides_ok(p.sdq, eq) ||
        !strides_ok(p.sdk, ek) || !strides_ok(p.sdv, ek)) {
        *why = "rows must start on 16-byte boundaries"; return false;
    }
    // P and dprobs rows are read in 16-byte chunks from their own start
    if ((p.Sq > 1 && p.sp[2] % 8 != 0) || (p.dprobs && p.Sq > 1 && p.sgp[2] % 8 != 0)) {
        *why = "probs and dprobs rows must start on 16-byte boundaries"; return false;
    }
    if (rows_broadcast(p.sq, p.Sq) || rows_broadcast(p.sp, p.Sq) || rows_broadcast(p.sgo, p.Sq) ||
        (p.dprobs && rows_broadcast(p.sgp, p.Sq)) || rows_broadcast(p.sk, p.Skv) || rows_broadcast(p.sv, p.Skv)) {
        *why = "an input's rows are broadcast (row stride 0): TMA tiles need distinct rows"; return false;
    }
    return true;
}

namespace {
template <int D, typename T>
cudaError_t launch_bwd_tc_t(const BwdProblem& p, cudaStream_t stream) {
    BwdIO io;
    std::memset(&io, 0, sizeof(io));
    io.q = p.q; io.sq0 = p.sq[0]; io.sq1 = p.sq[1]; io.sq2 = p.sq[2];
    io.k = p.k; io.sk0 = p.sk[0]; io.sk1 = p.sk[1]; io.sk2 = p.sk[2];
    io.v = p.v; io.sv0 = p.sv[0]; io.sv1 = p.sv[1]; io.sv2 = p.sv[2];
    io.p = p.p; io.sp0 = p.sp[0]; io.sp1 = p.sp[1]; io.sp2 = p.sp[2];
    io.go = p.dout; io.sgo0 = p.sgo[0]; io.sgo1 = p.sgo[1]; io.sgo2 = p.sgo[2];
    io.gp = p.dprobs; io.sgp0 = p.sgp[0]; io.sgp1 = p.sgp[1]; io.sgp2 = p.sgp[2];
    io.dq = p.dq; io.sdq0 = p.sdq[0]; io.sdq1 = p.sdq[1]; io.sdq2 = p.sdq[2];
    io.dk = p.dk; io.sdk0 = p.sdk[0]; io.sdk1 = p.sdk[1]; io.sdk2 = p.sdk[2];
    io.dv = p.dv; io.sdv0 = p.sdv[0]; io.sdv1 = p.sdv[1]; io.sdv2 = p.sdv[2];
    io.rowsum = p.rowsum;
    io.Hq = (int)p.Hq; io.group = (int)p.group; io.Sq = (int)p.Sq; io.Skv = (int)p.Skv;
    io.scale = p.scale;
    constexpr int smem = BwdKeysSmem<D>::kSmem, smem_rows = BwdRowsSmem<D>::kSmem;
    auto kr = bwd_tc_rows_kernel<D, T>;
    auto kk = bwd_tc_keys_kernel<D, T>;
    cudaError_t e = prepare_kernel(kr, smem_rows, false);
    if (e != cudaSuccess) return e;
    if ((e = prepare_kernel(kk, smem, false)) != cudaSuccess) return e;
    // tensor maps of the rows kernel's TMA operands ([B, H, S, X], 64-wide boxes)
    CUtensorMap mgo, mv, mk, mp, mg;
    BwdOrd ord;
    std::memset(&ord, 0, sizeof(ord));
    if (!make_map(&mgo, p.dtype, p.dout, p.Dv, p.Sq, p.Hq, p.B, p.sgo, 128, &ord.go) ||
        !make_map(&mv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, 64, &ord.v) ||
        !make_map(&mk, p.dtype, p.k, p.D, p.Skv, p.Hkv, p.B, p.sk, 64, &ord.k) ||
        !make_map(&mp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, 128, &ord.p))
        return cudaErrorNotSupported;
    if (p.dprobs) {
        if (!make_map(&mg, p.dtype, p.dprobs, p.Skv, p.Sq, p.Hq, p.B, p.sgp, 128, &ord.g)) return cudaErrorNotSupported;
    } else {
        mg = mp;  // never read
    }
    kr<<<dim3((unsigned)((p.Sq + 127) / 128), (unsigned)p.Hq, (unsigned)p.B), kBwdThreads, smem_rows, stream>>>(
        mgo, mv, mk, mp, mg, io, ord);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CUtensorMap kv, kgo, kq, kp, kg;
    BwdOrd ko;
    std::memset(&ko, 0, sizeof(ko));
    if (!make_map(&kv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, 128, &ko.v) ||
        !make_map(&kgo, p.dtype, p.dout, p.Dv, p.Sq, p.Hq, p.B, p.sgo, 64, &ko.go) ||
        !make_map(&kq, p.dtype, p.q, p.D, p.Sq, p.Hq, p.B, p.sq, 64, &ko.q) ||
        !make_map(&kp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, 64, &ko.p))
        return cudaErrorNotSupported;
    if (p.dprobs) {
        if (!make_map(&kg, p.dtype, p.dprobs, p.Skv, p.Sq, p.Hq, p.B, p.sgp, 64, &ko.g)) return cudaErrorNotSupported;
    } else {
        kg = kp;  // never read
    }
    kk<<<dim3((unsigned)((p.Skv + 127) / 128), (unsigned)p.Hkv, (unsigned)p.B), kBwdThreads, smem, stream>>>(
        kv, kgo, kq, kp, kg, io, ko);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_tc(const BwdProblem& p, cudaStream_t stream) {
    const char* why;
    if (!bwd_tc_supports(p, &why)) return cudaErrorNotSupported;
    if (p.dtype == kF16) return p.D == 64 ? launch_bwd_tc_t<64, __half>(p, stream) : launch_bwd_tc_t<128, __half>(p, stream);
    return p.D == 64 ? launch_bwd_tc_t<64, __nv_bfloat16>(p, stream) : launch_bwd_tc_t<128, __nv_bfloat16>(p, stream);
}

bool onesweep_supports(const Problem& p, const char** why) {
    if (!tc_supports(p, false, why)) return false;
    if (onesweep_cluster(p) == 0) {
        *why = "the one-sweep kernel keeps at most 32 live 128-key tiles per row block (8 CTAs x 4)";
        return false;
    }
    return true;
}

cudaError_t launch_tc(const Problem& p, int mode, cudaStream_t stream) {
    const char* why;
    if (mode < 1 || mode > 4) return cudaErrorNotSupported;
    if (mode == 4 ? !onesweep_supports(p, &why) : !tc_supports(p, mode == 3, &why)) return cudaErrorNotSupported;
    return p.dtype == kF16 ? launch_t<__half>(p, mode, stream) : launch_t<__nv_bfloat16>(p, mode, stream);
}

namespace {
// One thread waits on an mbarrier that nothing arrives at, through wait_bar:
// after kWaitLimitCycles the wait records role 15 in the device status word
// and returns false, and the kernel ends.
__global__ void selftest_wait_kernel() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)wait_bar(smem_u32(&bar), 0, &abort_flag, 15, 0);
}
}  // namespace

cudaError_t launch_selftest_wait(cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t status_read_and_clear(cudaStream_t stream, unsigned int* value) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(value, g_status_word, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace sdpa
