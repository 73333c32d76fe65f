// sdpa_tc.cu -- tcgen05 tensor-core kernel of the materialised-probability
// SDPA forward (fp16 / bf16, head dim 64 or 128).
//
// What it computes: FlagOS-OP PR #10 "feat: add sdpa_math operator" -- the
// math backend's (out, attn_probs): P = softmax(scale*QK^T + mask), O = P V,
// with a fully masked row giving P = O = 0.  P is normalised exactly through
// the row log-sum-exp, the identity of the page's "P800 exact-P fast path"
// update (P = exp(scale*QK^T - LSE)), which this kernel evaluates itself:
//
//   sweep 1  S_j = Q K_j^T on the tensor cores (TMEM accumulator), running
//            row max / sum of exp in the softmax warps -> lse per row;
//   sweep 2  S_j again, p = exp2(S_j*scale*log2e - lse*log2e) written once
//            as dtype into a 128B-swizzled shared tile that is both the A
//            operand of O += P_j V_j (tensor cores) and the source of the TMA
//            store of P; key tiles above a causal diagonal are never computed,
//            their P region is written with zeros by TMA stores.
//
// One CTA owns a 128-row query tile of one (batch, head); 8 warps:
//   warp 0      TMA producer (Q once; K tiles; then K/V tiles interleaved)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warp 2      TMA store issuer for P tiles (and the zero tiles)
//   warps 4..7  softmax / epilogue, one query row per thread (TMEM lane)
// TMEM: S double buffer (2 x 128 columns) + O (D columns) in one 512-column
// allocation.  Every mbarrier wait is bounded: a wait that runs out records
// itself in the device status word and the CTA unwinds without hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstring>
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

// The three outer tensor-map dimensions are stored in stride order; a packed
// code (2 bits per slot) says which logical dimension (1 = rows, 2 = head,
// 3 = batch) sits at tensor-map dim k+1, and pick() maps coordinates to it.
__device__ __forceinline__ int pick(uint32_t sel, int rows, int head, int batch) {
    return sel == 1 ? rows : (sel == 2 ? head : batch);
}

struct TcParams {
    int Sq, Skv, Hq, group, n_qtiles, causal;
    float c2;  // scale * log2(e)
    const void* mask;
    int mask_kind, mask_dtype;
    long long sm0, sm1, sm2;
    void* o;
    long long so0, so1, so2;
    float* lse;
    uint32_t ord_q, ord_k, ord_v, ord_p;
};

template <int D>
struct TcCfg {
    static constexpr int kChunks = D / 64;               // 128-byte (64-element) column chunks
    static constexpr int kTileBytes = 128 * D * 2;        // one Q / K / V tile
    static constexpr int kStages = (D == 64) ? 6 : 3;     // K/V ring depth
    static constexpr int kPBytes = 128 * 128 * 2;         // one P tile (2 chunks)
    static constexpr int kZeroBytes = 128 * 64 * 2;       // one zero chunk
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kTileBytes;
    static constexpr int kOffP = kOffKV + kStages * kTileBytes;
    static constexpr int kOffZ = kOffP + 2 * kPBytes;
    static constexpr int kOffBar = kOffZ + kZeroBytes;
    // barrier indices
    static constexpr int bQ = 0;
    static constexpr int bKVF = 1;
    static constexpr int bKVE = bKVF + kStages;
    static constexpr int bSF = bKVE + kStages;
    static constexpr int bSE = bSF + 2;
    static constexpr int bPF = bSE + 2;
    static constexpr int bPV = bPF + 2;
    static constexpr int bPS = bPV + 2;
    static constexpr int bO = bPS + 2;
    static constexpr int kBars = bO + 1;
    static constexpr int kSmem = kOffBar + kBars * 8 + 16 + 1024;  // + tmem slot, abort flag, alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kTmemO = 256;
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
    static __device__ __forceinline__ float load(const void* p) { return __half2float(*(const __half*)p); }
};
template <> struct Pack<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t two(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float load(const void* p) {
        return __bfloat162float(*(const __nv_bfloat16*)p);
    }
};

// Mask value of (row, key) in base-2 units to add to the score: 0, -inf, or
// an additive term.  Only called for rows < Sq and keys < Skv.
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

template <int D, typename T>
__global__ void __launch_bounds__(256, 1)
tc_twopass_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
                  const TcParams prm) {
    using C = TcCfg<D>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment of the shared-window offset (128B-swizzle atoms)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sQ = smem_u32(smem + C::kOffQ);
    const uint32_t sKV = smem_u32(smem + C::kOffKV);
    const uint32_t sP = smem_u32(smem + C::kOffP);
    const uint32_t sZ = smem_u32(smem + C::kOffZ);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int qt = prm.n_qtiles - 1 - (int)blockIdx.z;  // heaviest causal tiles first
    const int r0 = qt * 128;
    const int hk = h / prm.group;
    const int r_last = min(r0 + 127, prm.Sq - 1);
    const int n_all = (prm.Skv + 127) / 128;
    const int n_live = prm.causal ? (min(r_last, prm.Skv - 1) / 128 + 1) : n_all;

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        mbar_init(bar(C::bQ), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::bKVF + s), 1);
            mbar_init(bar(C::bKVE + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::bSF + i), 1);
            mbar_init(bar(C::bSE + i), 128);
            mbar_init(bar(C::bPF + i), 128);
            mbar_init(bar(C::bPV + i), 1);
            mbar_init(bar(C::bPS + i), 1);
        }
        mbar_init(bar(C::bO), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < C::kZeroBytes / 16; i += blockDim.x) st_shared_v4(sZ + i * 16, 0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        mbar_arrive_expect_tx(bar(C::bQ), C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c)
            tma_load_4d(sQ + c * 16384, &tm_q, bar(C::bQ), c * 64, pick(prm.ord_q & 3, r0, h, b),
                        pick((prm.ord_q >> 2) & 3, r0, h, b), pick((prm.ord_q >> 4) & 3, r0, h, b));
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
        for (int j = 0; j < n_live; ++j) load(&tm_k, prm.ord_k, j * 128);
        load(&tm_k, prm.ord_k, 0);
        for (int j = 1; j < n_live; ++j) {
            load(&tm_k, prm.ord_k, j * 128);
            load(&tm_v, prm.ord_v, (j - 1) * 128);
        }
        load(&tm_v, prm.ord_v, (n_live - 1) * 128);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBF16, false);
        constexpr uint32_t idesc_pv = idesc_f16(128, D, kBF16, true);
        wait_bar(bar(C::bQ), 0, abort_flag, 2, C::bQ);
        int it = 0, sc = 0;
        auto qk = [&]() {
            const int s = it % C::kStages;
            wait_bar(bar(C::bKVF + s), (it / C::kStages) & 1, abort_flag, 2, C::bKVF + s);
            const int buf = sc & 1;
            wait_bar(bar(C::bSE + buf), ((sc >> 1) & 1) ^ 1, abort_flag, 2, C::bSE + buf);
            tc_fence_after();
            const uint32_t d = tmem + buf * 128;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                tc_mma_f16(d, sw128_desc(sQ + off, 16, 1024), sw128_desc(sKV + s * C::kTileBytes + off, 16, 1024),
                           idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar(C::bKVE + s));
            tc_commit(bar(C::bSF + buf));
            ++it;
            ++sc;
        };
        auto pv = [&](int j) {
            const int pb = j & 1;
            wait_bar(bar(C::bPF + pb), (j >> 1) & 1, abort_flag, 2, C::bPF + pb);
            const int s = it % C::kStages;
            wait_bar(bar(C::bKVF + s), (it / C::kStages) & 1, abort_flag, 2, C::bKVF + s);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a_off = (kk / 4) * 16384 + (kk % 4) * 32;  // P: K-major, 16 keys per step
                const uint32_t b_off = kk * 2048;                         // V: N-major, 16 key rows per step
                tc_mma_f16(tmem + C::kTmemO, sw128_desc(sP + pb * C::kPBytes + a_off, 16, 1024),
                           sw128_desc(sKV + s * C::kTileBytes + b_off, 16384, 1024), idesc_pv,
                           (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar(C::bKVE + s));
            tc_commit(bar(C::bPV + pb));
            ++it;
        };
        for (int j = 0; j < n_live; ++j) qk();
        qk();
        for (int j = 1; j < n_live; ++j) {
            qk();
            pv(j - 1);
        }
        pv(n_live - 1);
        tc_commit(bar(C::bO));
    } else if (warp == 2 && lane == 0) {
        // ------------------------------------------------------------ P store issuer
        prefetch_tmap(&tm_p);
        const uint32_t o = prm.ord_p;
        for (int jz = n_live; jz < n_all; ++jz)
            for (int c = 0; c < 2; ++c)
                tma_store_4d(&tm_p, sZ, jz * 128 + c * 64, pick(o & 3, r0, h, b), pick((o >> 2) & 3, r0, h, b),
                             pick((o >> 4) & 3, r0, h, b));
        bulk_commit();
        for (int j = 0; j < n_live; ++j) {
            const int pb = j & 1;
            wait_bar(bar(C::bPF + pb), (j >> 1) & 1, abort_flag, 3, C::bPF + pb);
            for (int c = 0; c < 2; ++c)
                tma_store_4d(&tm_p, sP + pb * C::kPBytes + c * 16384, j * 128 + c * 64, pick(o & 3, r0, h, b),
                             pick((o >> 2) & 3, r0, h, b), pick((o >> 4) & 3, r0, h, b));
            bulk_commit();
            bulk_wait_read0();
            mbar_arrive(bar(C::bPS + pb));
        }
        bulk_wait0();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = threadIdx.x - 128;  // row within the tile == TMEM lane
        const int row = r0 + t;
        const bool row_ok = row < prm.Sq;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float c2 = prm.c2;
        const bool has_mask = prm.mask_kind != kMaskNone;
        float s[128];
        int sc = 0;

        auto load_s = [&](int role) {
            const int buf = sc & 1;
            wait_bar(bar(C::bSF + buf), (sc >> 1) & 1, abort_flag, role, C::bSF + buf);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + buf * 128 + c * 32, s + c * 32);
            tc_fence_before();
            mbar_arrive(bar(C::bSE + buf));
            ++sc;
        };
        // scale to base 2 and apply causal / ragged / user masking in place
        auto scale_mask = [&](int kv0) {
            const bool edge = (prm.causal && kv0 + 127 > r0) || (kv0 + 128 > prm.Skv) || !row_ok;
#pragma unroll
            for (int x = 0; x < 128; ++x) s[x] *= c2;
            if (edge || has_mask) {
#pragma unroll
                for (int x = 0; x < 128; ++x) {
                    const int key = kv0 + x;
                    float add = 0.f;
                    if (!row_ok || key >= prm.Skv || (prm.causal && key > row)) add = -CUDART_INF_F;
                    else if (has_mask) add = mask_term<T>(prm, b, h, row, key);
                    s[x] += add;
                }
            }
        };

        // sweep 1: row max and sum of exp2
        float m = -CUDART_INF_F, l = 0.f;
        for (int j = 0; j < n_live; ++j) {
            load_s(4);
            scale_mask(j * 128);
            float mt = -CUDART_INF_F;
#pragma unroll
            for (int x = 0; x < 128; ++x) mt = fmaxf(mt, s[x]);
            const float mn = fmaxf(m, mt);
            if (mn != -CUDART_INF_F) {
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
                for (int x = 0; x < 128; x += 4) {
                    acc0 += ex2(s[x] - mn);
                    acc1 += ex2(s[x + 1] - mn);
                    acc2 += ex2(s[x + 2] - mn);
                    acc3 += ex2(s[x + 3] - mn);
                }
                l = l * ex2(m - mn) + ((acc0 + acc1) + (acc2 + acc3));
                m = mn;
            }
        }
        const float lse2 = (m == -CUDART_INF_F) ? -CUDART_INF_F : m + log2f(l);
        const bool dead = lse2 == -CUDART_INF_F;

        // sweep 2: exact P into the swizzled shared tile
        for (int j = 0; j < n_live; ++j) {
            load_s(5);
            scale_mask(j * 128);
            const int pb = j & 1;
            const uint32_t ph = ((j >> 1) & 1) ^ 1;
            wait_bar(bar(C::bPV + pb), ph, abort_flag, 5, C::bPV + pb);
            wait_bar(bar(C::bPS + pb), ph, abort_flag, 5, C::bPS + pb);
            const uint32_t rowaddr = sP + pb * C::kPBytes + t * 128;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) p[e] = dead ? 0.f : ex2(s[u * 8 + e] - lse2);
                const uint32_t addr = rowaddr + (u / 8) * 16384 + (((u % 8) ^ (t % 8)) * 16);
                st_shared_v4(addr, Pack<T>::two(p[0], p[1]), Pack<T>::two(p[2], p[3]), Pack<T>::two(p[4], p[5]),
                             Pack<T>::two(p[6], p[7]));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(C::bPF + pb));
        }

        // epilogue: O from TMEM, direct 16-byte stores of this thread's row
        wait_bar(bar(C::bO), 0, abort_flag, 6, C::bO);
        tc_fence_after();
        T* orow = static_cast<T*>(prm.o) + b * prm.so0 + h * prm.so1 + (long long)row * prm.so2;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(tmem + lane_base + C::kTmemO + c * 32, ov);
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
        if (prm.lse && row_ok) prm.lse[((long long)b * prm.Hq + h) * prm.Sq + row] = dead ? lse2 : lse2 * kLn2;
    }

    // ------------------------------------------------------------ teardown
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
// of 64 x 128 rows, 128-byte swizzle.  The three outer dims are ordered by
// stride; `ord` receives the packed order code.
bool make_map(CUtensorMap* map, int dtype, const void* base, long long X, long long S, long long H, long long Bn,
              const int64_t* st /* [B, H, S] element strides */, uint32_t* ord) {
    auto fn = encode_fn();
    if (!fn) return false;
    struct Dim { long long ext, stride; int sel; };
    Dim d[3] = {{S, st[2], 1}, {H, st[1], 2}, {Bn, st[0], 3}};
    // extent-1 dims never move: give them a stride past everything else
    long long maxb = X;
    for (auto& x : d) if (x.ext > 1) maxb = std::max(maxb, x.stride * x.ext);
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
        box[k + 1] = d[k].sel == 1 ? 128 : 1;
        code |= (uint32_t)d[k].sel << (2 * k);
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *ord = code;
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool strides_ok(const int64_t* st, const int64_t* ext) {
    for (int i = 0; i < 3; ++i)
        if (ext[i] > 1 && st[i] % 8 != 0) return false;
    return true;
}

template <int D, typename T>
cudaError_t launch_twopass(const Problem& p, cudaStream_t stream) {
    using C = TcCfg<D>;
    CUtensorMap mq, mk, mv, mp;
    TcParams prm;
    std::memset(&prm, 0, sizeof(prm));
    if (!make_map(&mq, p.dtype, p.q, p.D, p.Sq, p.Hq, p.B, p.sq, &prm.ord_q) ||
        !make_map(&mk, p.dtype, p.k, p.D, p.Skv, p.Hkv, p.B, p.sk, &prm.ord_k) ||
        !make_map(&mv, p.dtype, p.v, p.Dv, p.Skv, p.Hkv, p.B, p.sv, &prm.ord_v) ||
        !make_map(&mp, p.dtype, p.p, p.Skv, p.Sq, p.Hq, p.B, p.sp, &prm.ord_p))
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
    auto kern = tc_twopass_kernel<D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)p.Hq, (unsigned)p.B, (unsigned)prm.n_qtiles);
    kern<<<grid, 256, C::kSmem, stream>>>(mq, mk, mv, mp, prm);
    return cudaGetLastError();
}

}  // namespace

bool tc_supports(const Problem& p, bool fused, const char** why) {
    if (fused) { *why = "the fused single-sweep kernel is not built yet"; return false; }
    if (p.dtype != kF16 && p.dtype != kBF16) { *why = "dtype must be f16 or bf16"; return false; }
    if (p.D != p.Dv || (p.D != 64 && p.D != 128)) { *why = "head dim must be 64 or 128 (D == Dv)"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (p.Sq >= (1ll << 31) || p.Skv >= (1ll << 31) || p.B > 65535 || p.Sq > 65535ll * 128) {
        *why = "sizes beyond the grid limits"; return false;
    }
    if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.p) || !aligned16(p.o)) {
        *why = "q, k, v, out and probs must be 16-byte aligned"; return false;
    }
    const int64_t eq[3] = {p.B, p.Hq, p.Sq}, ek[3] = {p.B, p.Hkv, p.Skv};
    if (!strides_ok(p.sq, eq) || !strides_ok(p.sk, ek) || !strides_ok(p.sv, ek) || !strides_ok(p.sp, eq) ||
        !strides_ok(p.so, eq)) {
        *why = "outer strides must be multiples of 8 elements (16 bytes)"; return false;
    }
    return true;
}

cudaError_t launch_tc(const Problem& p, bool fused, cudaStream_t stream) {
    const char* why;
    if (!tc_supports(p, fused, &why)) return cudaErrorNotSupported;
    if (p.dtype == kF16)
        return p.D == 64 ? launch_twopass<64, __half>(p, stream) : launch_twopass<128, __half>(p, stream);
    return p.D == 64 ? launch_twopass<64, __nv_bfloat16>(p, stream) : launch_twopass<128, __nv_bfloat16>(p, stream);
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
