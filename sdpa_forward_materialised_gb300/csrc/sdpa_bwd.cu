// sdpa_bwd.cu -- backward of the materialised-probability SDPA forward: the
// gradients for q, k and v when both outputs carry one (dout for O, dprobs
// for P), given the forward's probability map P.
//
// What it computes: FlagOS-OP PR #10 (overview, A1 item: the gradient flows
// through both outputs, dout and dprobs; "2026-10-07 update: P800 fused
// backward": dprobs goes through the exact softmax Jacobian of the
// materialised map and the query / key gradients of a GQA group are reduced
// back to its KV head).  Per (b, h, i), hk = h / (Hq / Hkv):
//     dP[i,j]  = dout[i,:] . v[hk,j,:] + dprobs[i,j]
//     rsum[i]  = sum_j P[i,j] dP[i,j]
//     dS[i,j]  = P[i,j] (dP[i,j] - rsum[i])
//     dq[i,:]  = scale sum_j dS[i,j] k[hk,j,:]
//     dk[hk,j,:] = scale sum_{h in group, i} dS[i,j] q[h,i,:]
//     dv[hk,j,:] = sum_{h in group, i} P[i,j] dout[h,i,:]
// Masked keys and fully masked rows have P = 0 and so no gradient.
//
// Two CUDA-core kernels, fp32 accumulation, outputs rounded to the dtype:
//   rows  one CTA per 32 query rows of one (b, h); four threads per row, each
//         owning a quarter of the head dim.  Two passes over 32-key tiles of
//         K and V staged in shared memory: the first forms rsum, the second
//         dS and dq.  rsum goes to the caller's buffer.
//   keys  one CTA per 32 keys of one (b, hk); four threads per key.  Walks
//         every query row of the group in staged tiles of 16 and accumulates
//         dk and dv in registers; no atomics, the GQA reduction stays inside
//         the CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace sdpa {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kTile = 32;     // keys per staged tile (rows kernel) / keys per CTA (keys kernel)
constexpr int kRowTile = 16;  // query rows per staged tile (keys kernel)

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld<__half>(const __half* p) { return __half2float(*p); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T> __device__ __forceinline__ void st(T* p, float x);
template <> __device__ __forceinline__ void st<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void st<__half>(__half* p, float x) { *p = __float2half_rn(x); }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// sum over the four threads of a row / key (adjacent lanes)
__device__ __forceinline__ float quad_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

// ---------------------------------------------------------------- rows kernel
// DQ = per-thread slice of the head dims (D / 4 and Dv / 4 rounded up, <= DQ).
template <typename T, int DQ>
__global__ void __launch_bounds__(kBwdThreads)
bwd_rows_kernel(const BwdProblem p) {
    extern __shared__ float sh[];
    float* ks = sh;                         // [kTile][D]
    float* vs = ks + kTile * p.D;           // [kTile][Dv]
    const int t = threadIdx.x, lr = t / 4, part = t % 4;
    const int b = blockIdx.z, h = blockIdx.y, hk = h / p.group;
    const int i = blockIdx.x * kTile + lr;  // query row
    const bool row_ok = i < p.Sq;
    const int dq0 = part * DQ, dv0 = part * DQ;  // this thread's dims [d0, d0 + DQ)

    const T* K = static_cast<const T*>(p.k) + b * p.sk[0] + hk * p.sk[1];
    const T* V = static_cast<const T*>(p.v) + b * p.sv[0] + hk * p.sv[1];
    const long long row_p = b * p.sp[0] + h * p.sp[1] + (long long)i * p.sp[2];
    const T* Pr = static_cast<const T*>(p.p) + row_p;
    const T* Gp = p.dprobs ? static_cast<const T*>(p.dprobs) + b * p.sgp[0] + h * p.sgp[1] + (long long)i * p.sgp[2]
                           : nullptr;
    // this thread's slice of dout[i, :]
    float go[DQ];
    {
        const T* G = static_cast<const T*>(p.dout) + b * p.sgo[0] + h * p.sgo[1] + (long long)i * p.sgo[2];
#pragma unroll
        for (int e = 0; e < DQ; ++e) go[e] = (row_ok && dv0 + e < p.Dv) ? ld(G + dv0 + e) : 0.f;
    }
    auto stage = [&](int j0) {
        __syncthreads();
        for (int x = t; x < kTile * p.D; x += kBwdThreads) {
            const int jj = x / p.D, d = x % p.D, j = j0 + jj;
            ks[x] = j < p.Skv ? ld(K + (long long)j * p.sk[2] + d) : 0.f;
        }
        for (int x = t; x < kTile * p.Dv; x += kBwdThreads) {
            const int jj = x / p.Dv, e = x % p.Dv, j = j0 + jj;
            vs[x] = j < p.Skv ? ld(V + (long long)j * p.sv[2] + e) : 0.f;
        }
        __syncthreads();
    };
    // dP[i, j] for a staged key jj (all four threads of the row get it)
    auto dprob = [&](int jj, int j) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < DQ; ++e)
            if (dv0 + e < p.Dv) a = fmaf(go[e], vs[jj * p.Dv + dv0 + e], a);
        a = quad_sum(a);
        if (Gp && row_ok) a += ld(Gp + j);
        return a;
    };

    // pass 1: rsum = sum_j P dP
    float rsum = 0.f;
    for (int j0 = 0; j0 < p.Skv; j0 += kTile) {
        stage(j0);
        for (int jj = 0; jj < kTile && j0 + jj < p.Skv; ++jj) {
            const int j = j0 + jj;
            const float dp = dprob(jj, j);
            const float pr = row_ok ? ld(Pr + j) : 0.f;
            rsum = fmaf(pr, dp, rsum);
        }
    }
    // pass 2: dS and dq
    float dq[DQ];
#pragma unroll
    for (int d = 0; d < DQ; ++d) dq[d] = 0.f;
    for (int j0 = 0; j0 < p.Skv; j0 += kTile) {
        stage(j0);
        for (int jj = 0; jj < kTile && j0 + jj < p.Skv; ++jj) {
            const int j = j0 + jj;
            const float dp = dprob(jj, j);
            const float pr = row_ok ? ld(Pr + j) : 0.f;
            const float ds = pr * (dp - rsum);
#pragma unroll
            for (int d = 0; d < DQ; ++d)
                if (dq0 + d < p.D) dq[d] = fmaf(ds, ks[jj * p.D + dq0 + d], dq[d]);
        }
    }
    if (row_ok) {
        T* Q = static_cast<T*>(p.dq) + b * p.sdq[0] + h * p.sdq[1] + (long long)i * p.sdq[2];
#pragma unroll
        for (int d = 0; d < DQ; ++d)
            if (dq0 + d < p.D) st(Q + dq0 + d, p.scale * dq[d]);
        if (part == 0) p.rowsum[((long long)b * p.Hq + h) * p.Sq + i] = rsum;
    }
}

// ---------------------------------------------------------------- keys kernel
template <typename T, int DQ>
__global__ void __launch_bounds__(kBwdThreads)
bwd_keys_kernel(const BwdProblem p) {
    extern __shared__ float sh[];
    float* qs = sh;                           // [kRowTile][D]
    float* gs = qs + kRowTile * p.D;          // [kRowTile][Dv]
    float* ps = gs + kRowTile * p.Dv;         // [kRowTile][kTile]  P
    float* hs = ps + kRowTile * kTile;        // [kRowTile][kTile]  dprobs
    float* rs = hs + kRowTile * kTile;        // [kRowTile]         rsum
    const int t = threadIdx.x, lj = t / 4, part = t % 4;
    const int b = blockIdx.z, hk = blockIdx.y;
    const int j0 = blockIdx.x * kTile, j = j0 + lj;
    const bool key_ok = j < p.Skv;
    const int d0 = part * DQ;

    // this thread's slice of v[hk, j, :]
    float vv[DQ];
    {
        const T* V = static_cast<const T*>(p.v) + b * p.sv[0] + hk * p.sv[1] + (long long)j * p.sv[2];
#pragma unroll
        for (int e = 0; e < DQ; ++e) vv[e] = (key_ok && d0 + e < p.Dv) ? ld(V + d0 + e) : 0.f;
    }
    float dk[DQ], dv[DQ];
#pragma unroll
    for (int d = 0; d < DQ; ++d) dk[d] = dv[d] = 0.f;

    const long long nrows = (long long)p.group * p.Sq;  // (head in group, i) pairs
    for (long long f0 = 0; f0 < nrows; f0 += kRowTile) {
        __syncthreads();
        // stage q, dout rows and the P / dprobs / rsum entries of this key block
        for (int x = t; x < kRowTile * p.D; x += kBwdThreads) {
            const int r = x / p.D, d = x % p.D;
            const long long f = f0 + r;
            float val = 0.f;
            if (f < nrows) {
                const int h = hk * p.group + (int)(f / p.Sq), i = (int)(f % p.Sq);
                val = ld(static_cast<const T*>(p.q) + b * p.sq[0] + h * p.sq[1] + (long long)i * p.sq[2] + d);
            }
            qs[x] = val;
        }
        for (int x = t; x < kRowTile * p.Dv; x += kBwdThreads) {
            const int r = x / p.Dv, e = x % p.Dv;
            const long long f = f0 + r;
            float val = 0.f;
            if (f < nrows) {
                const int h = hk * p.group + (int)(f / p.Sq), i = (int)(f % p.Sq);
                val = ld(static_cast<const T*>(p.dout) + b * p.sgo[0] + h * p.sgo[1] + (long long)i * p.sgo[2] + e);
            }
            gs[x] = val;
        }
        for (int x = t; x < kRowTile * kTile; x += kBwdThreads) {
            const int r = x / kTile, jj = x % kTile;
            const long long f = f0 + r;
            float pv = 0.f, hv = 0.f;
            if (f < nrows && j0 + jj < p.Skv) {
                const int h = hk * p.group + (int)(f / p.Sq), i = (int)(f % p.Sq);
                pv = ld(static_cast<const T*>(p.p) + b * p.sp[0] + h * p.sp[1] + (long long)i * p.sp[2] + j0 + jj);
                if (p.dprobs)
                    hv = ld(static_cast<const T*>(p.dprobs) + b * p.sgp[0] + h * p.sgp[1] + (long long)i * p.sgp[2] +
                            j0 + jj);
            }
            ps[x] = pv;
            hs[x] = hv;
        }
        if (t < kRowTile) {
            const long long f = f0 + t;
            float rv = 0.f;
            if (f < nrows) {
                const int h = hk * p.group + (int)(f / p.Sq), i = (int)(f % p.Sq);
                rv = p.rowsum[((long long)b * p.Hq + h) * p.Sq + i];
            }
            rs[t] = rv;
        }
        __syncthreads();
        for (int r = 0; r < kRowTile; ++r) {
            // dP[i, j] = dout[i] . v[j] + dprobs[i, j]
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < DQ; ++e)
                if (d0 + e < p.Dv) a = fmaf(gs[r * p.Dv + d0 + e], vv[e], a);
            a = quad_sum(a) + hs[r * kTile + lj];
            const float pr = ps[r * kTile + lj];
            const float ds = pr * (a - rs[r]);
#pragma unroll
            for (int d = 0; d < DQ; ++d) {
                if (d0 + d < p.D) dk[d] = fmaf(ds, qs[r * p.D + d0 + d], dk[d]);
                if (d0 + d < p.Dv) dv[d] = fmaf(pr, gs[r * p.Dv + d0 + d], dv[d]);
            }
        }
    }
    if (key_ok) {
        T* K = static_cast<T*>(p.dk) + b * p.sdk[0] + hk * p.sdk[1] + (long long)j * p.sdk[2];
        T* V = static_cast<T*>(p.dv) + b * p.sdv[0] + hk * p.sdv[1] + (long long)j * p.sdv[2];
#pragma unroll
        for (int d = 0; d < DQ; ++d) {
            if (d0 + d < p.D) st(K + d0 + d, p.scale * dk[d]);
            if (d0 + d < p.Dv) st(V + d0 + d, dv[d]);
        }
    }
}

template <typename T, int DQ>
cudaError_t launch_dq(const BwdProblem& p, cudaStream_t stream) {
    const size_t rows_smem = sizeof(float) * (size_t)kTile * (size_t)(p.D + p.Dv);
    const size_t keys_smem =
        sizeof(float) * ((size_t)kRowTile * (size_t)(p.D + p.Dv) + 2 * (size_t)kRowTile * kTile + kRowTile);
    auto kr = bwd_rows_kernel<T, DQ>;
    auto kk = bwd_keys_kernel<T, DQ>;
    cudaError_t e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rows_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)keys_smem);
    if (e != cudaSuccess) return e;
    if (p.Sq > 0) {
        dim3 grid((unsigned)((p.Sq + kTile - 1) / kTile), (unsigned)p.Hq, (unsigned)p.B);
        kr<<<grid, kBwdThreads, rows_smem, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.Skv > 0) {
        dim3 grid((unsigned)((p.Skv + kTile - 1) / kTile), (unsigned)p.Hkv, (unsigned)p.B);
        kk<<<grid, kBwdThreads, keys_smem, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_bwd_t(const BwdProblem& p, cudaStream_t stream) {
    const int64_t dmax = p.D > p.Dv ? p.D : p.Dv;
    if (dmax <= 64) return launch_dq<T, 16>(p, stream);
    if (dmax <= 128) return launch_dq<T, 32>(p, stream);
    return launch_dq<T, 64>(p, stream);
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem& p, cudaStream_t stream) {
    switch (p.dtype) {
        case kF32: return launch_bwd_t<float>(p, stream);
        case kF16: return launch_bwd_t<__half>(p, stream);
        case kBF16: return launch_bwd_t<__nv_bfloat16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdpa
