// sdpa_simt.cu -- CUDA-core (FFMA) kernel of the materialised-probability
// SDPA forward.  It serves every dtype (f32 / f16 / bf16), any head dim up to
// 256, any strides with a unit innermost stride, bool and additive masks and
// ragged sizes; it is the only family for f32 (tf32 tensor cores cannot meet
// f32 accuracy) and the fallback for layouts the tensor-core kernels reject.
//
// What it computes: FlagOS-OP PR #10 "feat: add sdpa_math operator" -- the
// math backend's (out, attn_probs), with P normalised exactly through the row
// log-sum-exp (the page's "P800 exact-P fast path" identity
// P = exp(scale*QK^T - LSE)).  Two sweeps over the keys:
//   sweep 1: scores -> running (max, sum) per row -> lse;
//   sweep 2: scores again -> p = exp(s - lse) -> P store, and O += p V.
// Fully masked rows have lse = -inf and give p = 0, hence P = O = 0.
//
// Work split: one CTA of 128 threads owns 16 query rows that share one
// key/value head (rows of the Hq/Hkv query heads of a GQA group are packed
// together, so K/V tiles are read once for the whole group) and walks the keys
// in tiles of 64.  All arithmetic is fp32; exponentials are base 2 with the
// scale folded into log2(e).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "internal.h"

namespace sdpa {
namespace {

constexpr int kThreads = 128;
constexpr int kRows = 16;   // query rows per CTA
constexpr int kTileK = 64;  // keys per tile
constexpr int kScoresPerThread = kRows * kTileK / kThreads;  // 8
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Merge two partial (max, sum) pairs of base-2 exponentials.
__device__ __forceinline__ void merge_ms(float& m, float& l, float m2, float l2) {
    const float mn = fmaxf(m, m2);
    if (mn == -CUDART_INF_F) return;  // both empty
    l = l * exp2f(m - mn) + l2 * exp2f(m2 - mn);
    m = mn;
}

struct RowInfo {
    int64_t h, i;  // query head and query position; h < 0 for padding rows
};

template <typename T, int kAccPerThread>
__global__ void __launch_bounds__(kThreads)
simt_kernel(const Problem p) {
    extern __shared__ float smem[];
    const int D = (int)p.D, Dv = (int)p.Dv;
    const int kw = (D > Dv ? D : Dv) + 1;           // padded row of the K/V tile
    float* qs = smem;                                // [kRows][D]
    float* kv = qs + kRows * D;                      // [kTileK][kw]
    float* ps = kv + kTileK * kw;                    // [kRows][kTileK]
    float* red_m = ps + kRows * kTileK;              // [4 warps][8]
    float* red_l = red_m + 32;                       // [4 warps][8]
    float* lse2 = red_l + 32;                        // [kRows]
    __shared__ RowInfo rows[kRows];

    const int t = threadIdx.x;
    const int64_t b = blockIdx.z, hk = blockIdx.y;
    const int64_t rows_total = p.group * p.Sq;       // flattened (head-in-group, i)
    const int64_t f0 = (int64_t)blockIdx.x * kRows;

    if (t < kRows) {
        const int64_t f = f0 + t;
        if (f < rows_total) {
            rows[t].h = hk * p.group + f / p.Sq;
            rows[t].i = f % p.Sq;
        } else {
            rows[t].h = -1;
            rows[t].i = 0;
        }
    }
    __syncthreads();

    const T* Q = static_cast<const T*>(p.q);
    const T* K = static_cast<const T*>(p.k) + b * p.sk[0] + hk * p.sk[1];
    const T* V = static_cast<const T*>(p.v) + b * p.sv[0] + hk * p.sv[1];

    // q rows -> shared (fp32)
    for (int e = t; e < kRows * D; e += kThreads) {
        const int r = e / D, d = e % D;
        float x = 0.f;
        if (rows[r].h >= 0) x = to_f(Q[b * p.sq[0] + rows[r].h * p.sq[1] + rows[r].i * p.sq[2] + d]);
        qs[e] = x;
    }

    // the largest query position in the CTA bounds the causal key range
    int64_t imax = -1;
    for (int r = 0; r < kRows; ++r)
        if (rows[r].h >= 0 && rows[r].i > imax) imax = rows[r].i;
    const int64_t key_end = p.causal ? (imax + 1 < p.Skv ? imax + 1 : p.Skv) : p.Skv;
    const int64_t ntiles = (key_end + kTileK - 1) / kTileK;

    const float c2 = p.scale * kLog2e;  // scale folded into base 2
    const int c = t % kTileK;           // key within the tile owned by this thread
    const int rbase = t / kTileK;       // rows rbase, rbase+2, ..., rbase+14

    // Score of (row r, key j) in base-2 units; -inf when masked or out of range.
    auto score = [&](int r, int64_t j) -> float {
        const RowInfo ri = rows[r];
        if (ri.h < 0 || j >= p.Skv) return -CUDART_INF_F;
        if (p.causal && j > ri.i) return -CUDART_INF_F;
        const float* qr = qs + r * D;
        const float* kr = kv + c * kw;
        float acc = 0.f;
        for (int d = 0; d < D; ++d) acc = fmaf(qr[d], kr[d], acc);
        float s = __fmul_rn(acc, c2);
        if (p.mask_kind != kMaskNone) {
            const int64_t off = b * p.sm[0] + ri.h * p.sm[1] + ri.i * p.sm[2] + j;
            if (p.mask_kind == kMaskBool) {
                if (static_cast<const unsigned char*>(p.mask)[off] == 0) s = -CUDART_INF_F;
            } else {
                float m;
                if (p.mask_dtype == kF32) m = static_cast<const float*>(p.mask)[off];
                else m = to_f(static_cast<const T*>(p.mask)[off]);
                s = __fmaf_rn(m, kLog2e, s);
            }
        }
        return s;
    };

    auto load_tile = [&](const T* base, const int64_t* st, int width, int64_t j0) {
        for (int e = t; e < kTileK * width; e += kThreads) {
            const int jj = e / width, d = e % width;
            const int64_t j = j0 + jj;
            kv[jj * kw + d] = (j < p.Skv) ? to_f(base[j * st[2] + d]) : 0.f;
        }
    };

    // ---------------- sweep 1: per-thread running (max, sum) ----------------
    float m_run[kScoresPerThread], l_run[kScoresPerThread];
#pragma unroll
    for (int u = 0; u < kScoresPerThread; ++u) { m_run[u] = -CUDART_INF_F; l_run[u] = 0.f; }

    for (int64_t kt = 0; kt < ntiles; ++kt) {
        const int64_t j0 = kt * kTileK;
        __syncthreads();
        load_tile(K, p.sk, D, j0);
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kScoresPerThread; ++u) {
            const float s = score(rbase + 2 * u, j0 + c);
            merge_ms(m_run[u], l_run[u], s, 1.f);
        }
    }

    // combine the 64 threads of each row: 32 lanes, then the two warps
    const int warp = t / 32, lane = t % 32;
#pragma unroll
    for (int u = 0; u < kScoresPerThread; ++u) {
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m_run[u], off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l_run[u], off);
            merge_ms(m_run[u], l_run[u], m2, l2);
        }
        if (lane == 0) { red_m[warp * 8 + u] = m_run[u]; red_l[warp * 8 + u] = l_run[u]; }
    }
    __syncthreads();
    if (t < kRows) {
        // row r = rbase + 2u lives in warps {2*rbase, 2*rbase+1}
        const int r = t, rb = r % 2, u = r / 2;
        float m = red_m[(2 * rb) * 8 + u], l = red_l[(2 * rb) * 8 + u];
        merge_ms(m, l, red_m[(2 * rb + 1) * 8 + u], red_l[(2 * rb + 1) * 8 + u]);
        const float v = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
        lse2[r] = v;
        if (p.lse && rows[r].h >= 0)
            p.lse[(b * p.Hq + rows[r].h) * p.Sq + rows[r].i] = (v == -CUDART_INF_F) ? v : v * kLn2;
    }
    __syncthreads();

    // ---------------- sweep 2: exact P, P store, O += P V ----------------
    float acc[kAccPerThread];
#pragma unroll
    for (int a = 0; a < kAccPerThread; ++a) acc[a] = 0.f;
    float row_lse[kScoresPerThread];
#pragma unroll
    for (int u = 0; u < kScoresPerThread; ++u) row_lse[u] = lse2[rbase + 2 * u];

    T* P = static_cast<T*>(p.p);
    const int64_t ptiles = (p.Skv + kTileK - 1) / kTileK;  // P is written over all keys
    for (int64_t kt = 0; kt < ptiles; ++kt) {
        const int64_t j0 = kt * kTileK;
        const bool live = kt < ntiles;
        if (live) {
            __syncthreads();
            load_tile(K, p.sk, D, j0);
            __syncthreads();
        }
#pragma unroll
        for (int u = 0; u < kScoresPerThread; ++u) {
            const int r = rbase + 2 * u;
            const int64_t j = j0 + c;
            float pr = 0.f;
            if (live && row_lse[u] != -CUDART_INF_F) {
                const float s = score(r, j);
                pr = exp2f(s - row_lse[u]);
            }
            const T pt = from_f<T>(pr);
            if (rows[r].h >= 0 && j < p.Skv)
                P[b * p.sp[0] + rows[r].h * p.sp[1] + rows[r].i * p.sp[2] + j] = pt;
            // a dead tile skipped the barrier above: other threads may still be
            // reading ps for the previous tile, and nothing reads it for this one
            if (live) ps[r * kTileK + c] = (j < p.Skv) ? to_f(pt) : 0.f;
        }
        if (!live) continue;  // the whole tile is above every causal diagonal here
        __syncthreads();
        load_tile(V, p.sv, Dv, j0);
        __syncthreads();
#pragma unroll
        for (int a = 0; a < kAccPerThread; ++a) {
            const int e = t + a * kThreads;
            if (e < kRows * Dv) {
                const int r = e / Dv, d = e % Dv;
                const float* pr = ps + r * kTileK;
                float x = acc[a];
                for (int jj = 0; jj < kTileK; ++jj) x = fmaf(pr[jj], kv[jj * kw + d], x);
                acc[a] = x;
            }
        }
    }

    T* O = static_cast<T*>(p.o);
#pragma unroll
    for (int a = 0; a < kAccPerThread; ++a) {
        const int e = t + a * kThreads;
        if (e < kRows * Dv) {
            const int r = e / Dv, d = e % Dv;
            if (rows[r].h >= 0)
                O[b * p.so[0] + rows[r].h * p.so[1] + rows[r].i * p.so[2] + d] = from_f<T>(acc[a]);
        }
    }
}

template <typename T, int kAcc>
cudaError_t launch_t(const Problem& p, cudaStream_t stream) {
    const int D = (int)p.D, Dv = (int)p.Dv;
    const int kw = (D > Dv ? D : Dv) + 1;
    const size_t smem = sizeof(float) * (size_t)(kRows * D + kTileK * kw + kRows * kTileK + 32 + 32 + kRows);
    auto kern = simt_kernel<T, kAcc>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t rows_total = p.group * p.Sq;
    dim3 grid((unsigned)((rows_total + kRows - 1) / kRows), (unsigned)p.Hkv, (unsigned)p.B);
    kern<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const Problem& p, cudaStream_t stream) {
    // accumulators per thread: kRows * Dv / kThreads, rounded up to a bucket
    if (p.Dv <= 64) return launch_t<T, 8>(p, stream);
    if (p.Dv <= 128) return launch_t<T, 16>(p, stream);
    return launch_t<T, 32>(p, stream);
}

}  // namespace

cudaError_t launch_simt(const Problem& p, cudaStream_t stream) {
    if (p.B > 65535 || p.Hkv > 65535) return cudaErrorInvalidConfiguration;
    switch (p.dtype) {
        case kF32: return launch_dtype<float>(p, stream);
        case kF16: return launch_dtype<__half>(p, stream);
        case kBF16: return launch_dtype<__nv_bfloat16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdpa
