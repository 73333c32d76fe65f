// sdpa_decode.cu -- materialised-probability SDPA forward for few query rows
// per key/value head (decode: Hq/Hkv * Sq <= 16 rows), split over the keys
// across a thread-block cluster.
//
// What it computes: FlagOS-OP PR #10 "feat: add sdpa_math operator" -- the
// math backend's (out, attn_probs) with P normalised exactly through the row
// log-sum-exp (the page's "P800 exact-P fast path" identity
// P = exp(scale*QK^T - LSE)); fully masked rows give P = O = 0.
//
// With a handful of query rows the work is bound by reading K and V once from
// HBM, and a 128-row tensor-core tile would be mostly empty.  So one cluster
// of C CTAs owns one (batch, key/value head) and all R = group * Sq query rows
// that read it; CTA rank c owns a contiguous chunk of the keys:
//   1. start asynchronous copies of the V chunk into shared memory; stage
//      the R query rows as fp32;
//   2. scores: one thread per key loads its K row straight into registers
//      (16-byte loads, eight in flight) and forms the R dot products (FFMA,
//      base-2 units, masking); per-row (max, sum of exp2) of the chunk;
//   3. cluster barrier; every CTA reads the C partial statistics through
//      distributed shared memory and forms the same lse per row;
//   4. P for the chunk (coalesced stores) and the partial O = P_chunk V_chunk
//      from the rounded P; cluster barrier;
//   5. CTA c sums its slice of the O columns over the cluster (distributed
//      shared memory) and stores O; a last cluster barrier keeps every CTA's
//      shared memory alive until all reads are done.
// No global workspace is used and every CTA reaches every cluster barrier.
// A CTA needs little shared memory (the V chunk, the scores, the partial O),
// so all clusters of a decode-sized call are resident at once and every K and
// V read of the call is issued in the first few microseconds.
//
// 16-bit calls with head dims of 32, 64, 128 or 256 take stream_decode_kernel
// instead (same split; K and V stream through a shared-memory ring, both
// products on the warp-level tensor-core instructions, one cluster exchange);
// SDPA_MATH_DECODE_KERNEL=cluster keeps them on decode_kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace sdpa {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = 16;     // query rows per (batch, kv head)
constexpr int kMaxCluster = 8;   // portable cluster size
constexpr int kSmemBudget = 160 * 1024;
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

// the two elements of a packed pair of 16-bit values
template <typename T> __device__ __forceinline__ float2 unpack2(uint32_t w);
template <> __device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<__half2*>(&w));
}
template <> __device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cluster barrier that publishes nothing (a CTA's shared memory stays alive
// until every peer is done with it): no wait for this thread's global stores.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
// Address of the same shared-memory word in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}
__device__ __forceinline__ float ld_peer(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

struct DecParams {
    const void* q; long long sq0, sq1, sq2;
    const void* k; long long sk0, sk1, sk2;
    const void* v; long long sv0, sv1, sv2;
    const void* mask; int mask_kind, mask_dtype; long long sm0, sm1, sm2;
    void* o; long long so0, so1, so2;
    void* p; long long sp0, sp1, sp2;
    float* lse;
    int Hq, Sq, Skv, D, Dv, group, rows, chunk, causal;
    float c2;  // scale * log2(e)
    int off_v, off_q, off_s, off_o, off_stat;  // shared-memory layout (bytes)
    // streaming kernel only
    int off_ring, off_pt, off_fac, off_part;
    int k_contig, v_contig;  // key / value rows back to back (row stride == head dim)
};

__device__ __forceinline__ void cp_async_wait_ring() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// Every committed group of this thread but the newest one is complete.
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// RM is a compile-time bound on the query rows (R <= RM), so the per-row
// accumulators of the score phase stay in registers.
template <typename T, int RM>
__global__ void __launch_bounds__(kThreads, RM <= 8 ? 4 : 3)
decode_kernel(const DecParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float lse_s[kMaxRows];
    __shared__ int row_h[kMaxRows], row_i[kMaxRows];

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const uint32_t crank = cluster_rank();
    const int C = (int)(gridDim.x);  // the cluster spans the x dimension
    const int b = blockIdx.z, hk = blockIdx.y;
    const int k0 = (int)crank * p.chunk;
    const int n = max(0, min(p.Skv, k0 + p.chunk) - k0);  // keys of this CTA (may be 0)
    const int R = p.rows, D = p.D, Dv = p.Dv;

    uint8_t* vs = smem + p.off_v;                             // [n][Dv] V chunk (dtype)
    float* qs = reinterpret_cast<float*>(smem + p.off_q);     // [R][D] query rows (fp32)
    float* ss = reinterpret_cast<float*>(smem + p.off_s);     // [R][chunk] scores, then rounded P
    float* op = reinterpret_cast<float*>(smem + p.off_o);     // [R][Dv] partial O
    float* st = reinterpret_cast<float*>(smem + p.off_stat);  // [R][2] chunk (max, sum)

    // ---- 1. loads in the order they are needed: the query rows and the first
    // 128 bytes of this thread's K row into registers, then the V chunk
    // (asynchronous copies, needed last)
    const T* K = static_cast<const T*>(p.k) + b * p.sk0 + hk * p.sk1 + (long long)k0 * p.sk2;
    const T* V = static_cast<const T*>(p.v) + b * p.sv0 + hk * p.sv1 + (long long)k0 * p.sv2;
    float qv[RM];  // elements t, t + 256, ... of the [R][D] query block (R * D <= RM * 256)
#pragma unroll
    for (int i = 0; i < RM; ++i) {
        const int e = t + kThreads * i;
        qv[i] = 0.f;
        if (e < R * D) {
            const int r = e / D, d = e % D;
            const T* qr = static_cast<const T*>(p.q) + b * p.sq0 + (long long)(hk * p.group + r / p.Sq) * p.sq1 +
                          (long long)(r % p.Sq) * p.sq2;
            qv[i] = to_f(qr[d]);
        }
    }
    const uint8_t* krow = reinterpret_cast<const uint8_t*>(K + (long long)t * p.sk2);
    const int kbytes = D * (int)sizeof(T);
    uint4 kx[8];
    if (t < n) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (16 * u < kbytes) kx[u] = __ldg(reinterpret_cast<const uint4*>(krow + 16 * u));
    }
    {
        const int uv = Dv * (int)sizeof(T) / 16;  // 16-byte units per V row
        for (int u = t; u < n * uv; u += kThreads) {
            const int r = u / uv, c = u % uv;
            cp_async16(vs + 16 * u, reinterpret_cast<const uint8_t*>(V + r * p.sv2) + 16 * c);
        }
        cp_async_commit();
    }
    if (t < R) {
        row_h[t] = hk * p.group + t / p.Sq;
        row_i[t] = t % p.Sq;
    }
#pragma unroll
    for (int i = 0; i < RM; ++i)
        if (t + kThreads * i < R * D) qs[t + kThreads * i] = qv[i];
    __syncthreads();

    // ---- 2. scores: thread j owns key k0 + j and reads its K row straight
    // into registers, 128 bytes (eight 16-byte loads in flight) per batch;
    // the first batch was issued above
    if (t < n) {
        constexpr int kE = 16 / (int)sizeof(T);  // elements per 16-byte unit
        float acc[RM];
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] = 0.f;
        for (int b0 = 0; b0 < kbytes; b0 += 128) {
            if (b0 > 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (b0 + 16 * u < kbytes) kx[u] = __ldg(reinterpret_cast<const uint4*>(krow + b0 + 16 * u));
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (b0 + 16 * u >= kbytes) break;
                const int d = (b0 + 16 * u) / (int)sizeof(T);
                if constexpr (sizeof(T) == 4) {
                    const float4 kk = make_float4(__uint_as_float(kx[u].x), __uint_as_float(kx[u].y),
                                                  __uint_as_float(kx[u].z), __uint_as_float(kx[u].w));
#pragma unroll
                    for (int r = 0; r < RM; ++r)
                        if (r < R) {
                            const float4 qq = *reinterpret_cast<const float4*>(&qs[r * D + d]);
                            float a = acc[r];
                            a = fmaf(qq.x, kk.x, a);
                            a = fmaf(qq.y, kk.y, a);
                            a = fmaf(qq.z, kk.z, a);
                            a = fmaf(qq.w, kk.w, a);
                            acc[r] = a;
                        }
                } else {
                    static_assert(kE == 8, "16-bit elements");
                    const float2 k01 = unpack2<T>(kx[u].x), k23 = unpack2<T>(kx[u].y);
                    const float2 k45 = unpack2<T>(kx[u].z), k67 = unpack2<T>(kx[u].w);
#pragma unroll
                    for (int r = 0; r < RM; ++r)
                        if (r < R) {
                            const float4 qa = *reinterpret_cast<const float4*>(&qs[r * D + d]);
                            const float4 qb = *reinterpret_cast<const float4*>(&qs[r * D + d + 4]);
                            float a = acc[r];
                            a = fmaf(qa.x, k01.x, a);
                            a = fmaf(qa.y, k01.y, a);
                            a = fmaf(qa.z, k23.x, a);
                            a = fmaf(qa.w, k23.y, a);
                            a = fmaf(qb.x, k45.x, a);
                            a = fmaf(qb.y, k45.y, a);
                            a = fmaf(qb.z, k67.x, a);
                            a = fmaf(qb.w, k67.y, a);
                            acc[r] = a;
                        }
                }
            }
        }
        const int key = k0 + t;
#pragma unroll
        for (int r = 0; r < RM; ++r)
            if (r < R) {
                float s = __fmul_rn(acc[r], p.c2);
                if (p.causal && key > row_i[r]) s = -CUDART_INF_F;
                if (p.mask_kind != kMaskNone) {
                    const long long off = b * p.sm0 + row_h[r] * p.sm1 + (long long)row_i[r] * p.sm2 + key;
                    if (p.mask_kind == kMaskBool) {
                        if (static_cast<const unsigned char*>(p.mask)[off] == 0) s = -CUDART_INF_F;
                    } else {
                        const float m = p.mask_dtype == kF32 ? static_cast<const float*>(p.mask)[off]
                                                             : to_f(static_cast<const T*>(p.mask)[off]);
                        s = __fmaf_rn(m, kLog2e, s);
                    }
                }
                ss[r * p.chunk + t] = s;
            }
    }
    __syncthreads();

    // per-row (max, sum of exp2) of the chunk: one warp per row
    for (int r = warp; r < R; r += kThreads / 32) {
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

    // ---- 3. the cluster's statistics -> the same lse in every CTA
    cluster_sync();
    if (t < R) {
        float mc[kMaxCluster], lc[kMaxCluster];  // all peer loads first, then the merge
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) {
                mc[c] = ld_peer(peer_addr(&st[2 * t], (uint32_t)c));
                lc[c] = ld_peer(peer_addr(&st[2 * t + 1], (uint32_t)c));
            }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) m = fmaxf(m, mc[c]);
        float l = 0.f;
        if (m != -CUDART_INF_F) {
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                if (c < C && mc[c] != -CUDART_INF_F) l += lc[c] * exp2f(mc[c] - m);
        }
        lse_s[t] = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
    }
    __syncthreads();

    // ---- 4. P for the chunk, rounded to the dtype and kept for P V (stored to
    // global memory after the next cluster barrier, whose release then has
    // no global stores of this thread to wait for)
    for (int e = t; e < R * n; e += kThreads) {
        const int r = e / n, j = e % n;
        const float L = lse_s[r];
        const float pr = (L == -CUDART_INF_F) ? 0.f : exp2f(ss[r * p.chunk + j] - L);
        ss[r * p.chunk + j] = to_f(from_f<T>(pr));
    }
    cp_async_wait_all();
    __syncthreads();
    // partial O = P_chunk V_chunk; a thread item is (row, pair of columns)
    // (Dv is even: V rows are 16-byte multiples)
    const int dv2 = Dv / 2;
    for (int e = t; e < R * dv2; e += kThreads) {
        const int r = e / dv2, d = 2 * (e % dv2);
        const float* pr = ss + r * p.chunk;
        float a0 = 0.f, a1 = 0.f;
        for (int j = 0; j < n; ++j) {
            float2 vv;
            if constexpr (sizeof(T) == 4) vv = *reinterpret_cast<const float2*>(vs + (j * Dv + d) * 4);
            else vv = unpack2<T>(*reinterpret_cast<const uint32_t*>(vs + (j * Dv + d) * 2));
            a0 = fmaf(pr[j], vv.x, a0);
            a1 = fmaf(pr[j], vv.y, a1);
        }
        *reinterpret_cast<float2*>(&op[r * Dv + d]) = make_float2(a0, a1);
    }

    // ---- 5. sum this CTA's slice of the O columns over the cluster; store P
    cluster_sync();
    for (int e = t; e < R * n; e += kThreads) {
        const int r = e / n, j = e % n;
        T* prow = static_cast<T*>(p.p) + b * p.sp0 + row_h[r] * p.sp1 + (long long)row_i[r] * p.sp2;
        prow[k0 + j] = from_f<T>(ss[r * p.chunk + j]);
    }
    const int cols = (Dv + C - 1) / C;
    const int c0 = (int)crank * cols, c1 = min(Dv, c0 + cols);
    for (int e = t; e < R * max(0, c1 - c0); e += kThreads) {
        const int r = e / (c1 - c0), d = c0 + e % (c1 - c0);
        float part[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) part[c] = ld_peer(peer_addr(&op[r * Dv + d], (uint32_t)c));
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) acc += part[c];
        const bool dead = lse_s[r] == -CUDART_INF_F;
        T* orow = static_cast<T*>(p.o) + b * p.so0 + row_h[r] * p.so1 + (long long)row_i[r] * p.so2;
        orow[d] = from_f<T>(dead ? 0.f : acc);
    }
    if (crank == 0 && p.lse && t < R) {
        const float L = lse_s[t];
        p.lse[((long long)b * p.Hq + row_h[t]) * p.Sq + row_i[t]] = (L == -CUDART_INF_F) ? L : L * kLn2;
    }
    cluster_sync_relaxed();  // no CTA leaves while a peer may still read its shared memory
}



// ---------------------------------------------------------------------------
// Streaming decode kernel (16-bit inputs; head dims of 32, 64, 128 or 256).
//
// The cluster split of decode_kernel (one cluster per (batch, key/value head),
// CTA rank c owns a contiguous chunk of keys), with another data path inside
// the CTA, in two warp groups one 32-key piece apart:
//   * warps 0-3 stream K through a two-slot ring (two pieces ahead) and form
//     the partial scores S^T = K_piece Q^T of piece i (two k-groups) in one of
//     two shared buffers;
//   * warps 4-7 stream V through a three-slot ring (two pieces ahead) and,
//     for piece i - 1, run the masking and the chunk's online softmax (one
//     warp per row and one lane per key keep the running (max, sum); P~ =
//     exp2(s - running max), rounded to the input dtype, and the rescale
//     factors go to shared memory; the scores stay there for P) and
//     accumulate O += P~ V, rescaling O whenever the max grew;
//   * the groups pass the score buffers back and forth through double-
//     buffered named barriers (bar.arrive by the producing group, bar.sync by
//     the consuming one); each group waits only for its own asynchronous
//     copies;
//   * copies are 16-byte cp.async (consecutive threads on consecutive bytes of
//     a row), each 16-byte unit of a row placed at unit u ^ f(row), an XOR
//     swizzle that makes the 8-row matrix loads conflict-free;
//   * both products run on the tensor cores with the warp-level
//     mma.sync.m16n8k16 (fp16 / bf16 operands, fp32 accumulation): 16 keys by
//     8 query rows per score instruction, the query rows padded to 16 and 8
//     value columns per output instruction;
//   * one cluster barrier publishes every CTA's (max, sum) and partial O.
//     Each CTA then forms the same lse, writes its P = exp2(s - lse) and sums
//     its slice of the O columns over the cluster, the partial of CTA c
//     weighted by exp2(max_c - lse).
// ---------------------------------------------------------------------------
constexpr int kStreamTK = 32;   // keys per piece (one per lane in the row statistics)
constexpr int kPthPitch = kStreamTK + 8;  // P~ tile row pitch (elements): conflict-free fragment loads
constexpr int kKSlots = 2, kVSlots = 3;   // K / V ring slots (32-key pieces)
constexpr int kGroupThreads = 128;        // each of the two warp groups
constexpr int kBarGroup = 1, kBarFull = 2, kBarFree = 4;  // named barrier ids: copy group; [2] P~ ready; [2] P~ used
constexpr int kBarPV = 6;                                  // P V group

// Physical 16-byte unit of logical unit u in row `row` of a tile whose rows
// hold `units` units (4, 8, 16 or 32): eight consecutive rows read at the same
// logical unit land in eight different 16-byte bank groups.
__device__ __forceinline__ int swz(int row, int u, int units) {
    return units >= 8 ? (u ^ (row & 7)) : (u ^ ((row >> 1) & 3));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr) : "memory");
}

// c (16 x 8, fp32) += a (16 x 16, row) * b (16 x 8, col) in the operand dtype T.
template <typename T> __device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);
template <> __device__ __forceinline__ void mma16816<__half>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Every thread of one warp group: start its share of the 16-byte copies of
// the K rows (issue_k) or the V rows (issue_v) of piece `piece` of the chunk
// into a ring slot, each 16-byte unit u of row r at unit u ^ f(r), and commit
// them as one group.  V rows past the chunk's end get zeros (copies with no
// source bytes), so P~ V never multiplies a zero by stale shared memory.
template <typename T>
__device__ __forceinline__ void issue_rows(const T* X, long long sx, bool contig, int units, int j0, int tk,
                                           int rows, uint8_t* slot, int ta) {
    const int lu = __ffs(units) - 1;
    // rows back to back (row stride == head dim): the piece is one contiguous
    // block and unit c of it sits at byte 16 c
    const uint8_t* xp = reinterpret_cast<const uint8_t*>(X + (long long)j0 * sx);
    for (int c = ta; c < rows * units; c += kGroupThreads) {
        const int r = c >> lu, u = c & (units - 1);
        uint8_t* dst = slot + 16 * (r * units + swz(r, u, units));
        if (r < tk) {
            cp_async16(dst, contig ? xp + 16 * c : reinterpret_cast<const uint8_t*>(X + (long long)(j0 + r) * sx) + 16 * u);
        } else {
            const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(d), "l"(X) : "memory");
        }
    }
    cp_async_commit();
}
template <typename T>
__device__ __forceinline__ void issue_k(const DecParams& p, const T* K, int piece, int n, uint8_t* slot, int ta) {
    const int j0 = piece * kStreamTK, tk = min(kStreamTK, n - j0);
    issue_rows(K, p.sk2, p.k_contig != 0, p.D * (int)sizeof(T) / 16, j0, tk, tk, slot, ta);
}
template <typename T>
__device__ __forceinline__ void issue_v(const DecParams& p, const T* V, int piece, int n, uint8_t* slot, int ta) {
    const int j0 = piece * kStreamTK, tk = min(kStreamTK, n - j0);
    issue_rows(V, p.sv2, p.v_contig != 0, p.Dv * (int)sizeof(T) / 16, j0, tk, kStreamTK, slot, ta);
}

// Named barriers (immediate ids, so the kernel reserves only those it uses):
// bar.sync waits, bar.arrive only counts; every warp of a group executes them.
template <int ID, int N> __device__ __forceinline__ void nbar_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}
template <int ID, int N> __device__ __forceinline__ void nbar_arrive() {
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(N) : "memory");
}
// the two-slot handshakes between the warp groups, by the parity of the piece
__device__ __forceinline__ void full_arrive(int i) {
    if (i & 1) nbar_arrive<kBarFull + 1, 2 * kGroupThreads>();
    else nbar_arrive<kBarFull, 2 * kGroupThreads>();
}
__device__ __forceinline__ void full_sync(int i) {
    if (i & 1) nbar_sync<kBarFull + 1, 2 * kGroupThreads>();
    else nbar_sync<kBarFull, 2 * kGroupThreads>();
}
__device__ __forceinline__ void free_arrive(int i) {
    if (i & 1) nbar_arrive<kBarFree + 1, 2 * kGroupThreads>();
    else nbar_arrive<kBarFree, 2 * kGroupThreads>();
}
__device__ __forceinline__ void free_sync(int i) {
    if (i & 1) nbar_sync<kBarFree + 1, 2 * kGroupThreads>();
    else nbar_sync<kBarFree, 2 * kGroupThreads>();
}

template <typename T, int RM>
__global__ void __launch_bounds__(kThreads, RM <= 4 ? 4 : 2)
stream_decode_kernel(const DecParams p) {
    static_assert(sizeof(T) == 2, "16-bit inputs");
    constexpr int NT = RM > 8 ? 2 : 1;  // 8-row tiles of query rows in the score product
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float m_run[kMaxRows], l_run[kMaxRows], alpha_s[kMaxRows], lse_s[kMaxRows];
    __shared__ int row_h[kMaxRows], row_i[kMaxRows];

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const int g = lane >> 2, cc = lane & 3;  // fragment row / column pair of this lane
    const int mi = lane >> 3, r8 = lane & 7;  // this lane's matrix / row in an 8x8 matrix load
    const bool copy_group = warp < 4;
    const uint32_t crank = cluster_rank();
    const int C = (int)gridDim.x;  // the cluster spans the x dimension
    const int b = blockIdx.z, hk = blockIdx.y;
    const int k0 = (int)crank * p.chunk;
    const int n = max(0, min(p.Skv, k0 + p.chunk) - k0);  // keys of this CTA (may be 0)
    const int R = p.rows, D = p.D, Dv = p.Dv;
    const int npieces = (n + kStreamTK - 1) / kStreamTK;
    const int uk = D * (int)sizeof(T) / 16, uv = Dv * (int)sizeof(T) / 16;
    const int kbytes = kStreamTK * uk * 16, vbytes = kStreamTK * uv * 16;

    uint8_t* kring = smem + p.off_ring;               // [kKSlots][32 rows of K]
    uint8_t* vring = kring + kKSlots * kbytes;        // [kVSlots][32 rows of V]
    float* ss = reinterpret_cast<float*>(smem + p.off_s);      // [R][chunk] scores (base 2, masked)
    T* pth = reinterpret_cast<T*>(smem + p.off_pt);            // [16][kPthPitch] P~ of a piece
    float* part = reinterpret_cast<float*>(smem + p.off_part); // [2][2][RM][32] k-group partial scores of a piece
    float* op = reinterpret_cast<float*>(smem + p.off_ring);   // [R][Dv] partial O (the rings, after the loop)
    float* st = reinterpret_cast<float*>(smem + p.off_stat);   // [R][2] chunk (max, sum)
    float* fac = reinterpret_cast<float*>(smem + p.off_fac);   // [R][C] weight of each CTA's partial O

    const T* K = static_cast<const T*>(p.k) + b * p.sk0 + hk * p.sk1 + (long long)k0 * p.sk2;
    const T* V = static_cast<const T*>(p.v) + b * p.sv0 + hk * p.sv1 + (long long)k0 * p.sv2;

    // K (warps 0-3) and V (warps 4-7) of pieces 0 and 1
    for (int pc = 0; pc < 2; ++pc) {
        if (pc >= npieces) cp_async_commit();
        else if (copy_group) issue_k(p, K, pc, n, kring + pc * kbytes, t);
        else issue_v(p, V, pc, n, vring + pc * vbytes, t - kGroupThreads);
    }
    if (t < R) {
        row_h[t] = hk * p.group + t / p.Sq;
        row_i[t] = t % p.Sq;
        m_run[t] = -CUDART_INF_F;
        l_run[t] = 0.f;
    }
    for (int e = t; e < 16 * kPthPitch; e += kThreads) pth[e] = from_f<T>(0.f);  // rows past R stay zero
    __syncthreads();

    // the output product: warp 4 + w owns value-column tiles [ntw w, ntw (w + 1))
    const int nvt = Dv / 8;                  // 8-column tiles
    const int ntw = nvt >= 4 ? nvt / 4 : 1;  // tiles per warp: 1, 2, 4 or 8
    const bool pv_warp = !copy_group && warp - 4 < (nvt >= 4 ? 4 : nvt);

    if (copy_group) {
        // ---- warps 0-3: K copies and S^T = K Q^T, one piece ahead of the
        // statistics and the output product.  Warp w takes key tile w & 1 and
        // k-group w >> 1 (half the k-steps, two accumulators); its Q^T
        // fragments stay in registers.
        const int mt = warp & 1, kg = warp >> 1;
        const int per = D / 32;  // k-steps per group: 1, 2, 4 or 8
        uint32_t qb[NT][8][2];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                qb[i][s][0] = qb[i][s][1] = 0u;
                const int qr = 8 * i + g;
                if (s < per && qr < R) {
                    const unsigned short* qrow = reinterpret_cast<const unsigned short*>(
                        static_cast<const T*>(p.q) + b * p.sq0 + (long long)(hk * p.group + qr / p.Sq) * p.sq1 +
                        (long long)(qr % p.Sq) * p.sq2);
                    const int d = 16 * (kg * per + s) + 2 * cc;
                    qb[i][s][0] = (uint32_t)qrow[d] | ((uint32_t)qrow[d + 1] << 16);
                    qb[i][s][1] = (uint32_t)qrow[d + 8] | ((uint32_t)qrow[d + 9] << 16);
                }
            }
        const int key = 16 * mt + (mi & 1) * 8 + r8;  // this lane's row address for the K matrices
        for (int i = 0; i < npieces; ++i) {
            // this thread's K copies of piece i have landed (those of piece
            // i + 1 may still be in flight); the group barrier shares everyone's
            cp_async_wait_all_but_one();
            nbar_sync<kBarGroup, kGroupThreads>();
            // the partial-score buffer of piece i - 2 is free once its statistics are done
            if (i >= 2) free_sync(i);
            const uint32_t kslot = static_cast<uint32_t>(__cvta_generic_to_shared(kring + (i & 1) * kbytes));
            float* pp = part + (i & 1) * 2 * RM * kStreamTK;
            {
                float c[2][NT][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < NT; ++q) c[h][q][0] = c[h][q][1] = c[h][q][2] = c[h][q][3] = 0.f;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    if (s >= per) break;
                    uint32_t a[4];
                    ldsm_x4(kslot + 16 * (key * uk + swz(key, 2 * (kg * per + s) + (mi >> 1), uk)), a[0], a[1], a[2], a[3]);
#pragma unroll
                    for (int q = 0; q < NT; ++q) mma16816<T>(c[s & 1][q], a, qb[q][s][0], qb[q][s][1]);
                }
#pragma unroll
                for (int q = 0; q < NT; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = 8 * q + 2 * cc + (e & 1), kk = 16 * mt + g + 8 * (e >> 1);
                        if (row < R) pp[(kg * RM + row) * kStreamTK + kk] = c[0][q][e] + c[1][q][e];
                    }
            }
            nbar_sync<kBarGroup, kGroupThreads>();  // every warp is done with this K slot
            // K of piece i + 2 into this piece's K slot (its scores are done)
            if (i + 2 < npieces) issue_k(p, K, i + 2, n, kring + (i & 1) * kbytes, t);
            else cp_async_commit();
            full_arrive(i);
        }
        // the statistics' last releases
        for (int i = max(0, npieces - 2); i < npieces; ++i) free_sync(i);
        cp_async_wait_all();
    } else {
        // ---- warps 4-7: V copies, the masking and online statistics (one
        // warp per row, one lane per key) and O += P~ V (rows g and g + 8 of
        // each of this warp's column tiles), one piece behind the scores
        const int wb = warp - 4;
        float oc[8][4];
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) oc[q][e] = 0.f;
        for (int i = 0; i < npieces; ++i) {
            // this thread's V copies of piece i have landed (those of piece
            // i + 1 may still be in flight); the group barrier shares everyone's
            // and ends every warp's P V of piece i - 1, so V of piece i + 2
            // can take that piece's slot
            cp_async_wait_all_but_one();
            nbar_sync<kBarPV, kGroupThreads>();
            if (i + 2 < npieces) issue_v(p, V, i + 2, n, vring + ((i + 2) % kVSlots) * vbytes, t - kGroupThreads);
            else cp_async_commit();
            full_sync(i);
            {
                const int j0 = i * kStreamTK, tk = min(kStreamTK, n - j0);
                const float* pp = part + (i & 1) * 2 * RM * kStreamTK;
                for (int r = wb; r < R; r += 4) {
                    float sv = -CUDART_INF_F;
                    if (lane < tk) {
                        const int kglob = k0 + j0 + lane;
                        const float* pr = pp + r * kStreamTK + lane;
                        sv = __fmul_rn(pr[0] + pr[RM * kStreamTK], p.c2);
                        if (p.causal && kglob > row_i[r]) sv = -CUDART_INF_F;
                        if (p.mask_kind != kMaskNone) {
                            const long long off = b * p.sm0 + row_h[r] * p.sm1 + (long long)row_i[r] * p.sm2 + kglob;
                            if (p.mask_kind == kMaskBool) {
                                if (static_cast<const unsigned char*>(p.mask)[off] == 0) sv = -CUDART_INF_F;
                            } else {
                                const float m = p.mask_dtype == kF32 ? static_cast<const float*>(p.mask)[off]
                                                                     : to_f(static_cast<const T*>(p.mask)[off]);
                                sv = __fmaf_rn(m, kLog2e, sv);
                            }
                        }
                        ss[r * p.chunk + j0 + lane] = sv;
                    }
                    float mp = sv;
                    for (int o = 16; o > 0; o >>= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
                    const float mo = m_run[r];
                    const float mn = fmaxf(mo, mp);
                    const float ms = mn == -CUDART_INF_F ? 0.f : mn;  // a row with no visible key yet adds zeros
                    const float e = ptx::ex2(sv - ms);                 // sv = -inf gives 0
                    float sum = e;
                    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                    pth[r * kPthPitch + lane] = from_f<T>(e);
                    if (lane == 0) {
                        const float al = ptx::ex2(mo - ms);
                        alpha_s[r] = al;
                        m_run[r] = mn;
                        l_run[r] = l_run[r] * al + sum;
                    }
                }
            }
            free_arrive(i);                     // the partial scores of piece i are read
            nbar_sync<kBarPV, kGroupThreads>();  // P~ and the rescale factors are complete
            if (pv_warp) {
                const float a_lo = g < R ? alpha_s[g] : 0.f, a_hi = g + 8 < R ? alpha_s[g + 8] : 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (q < ntw) {
                        oc[q][0] *= a_lo; oc[q][1] *= a_lo;
                        oc[q][2] *= a_hi; oc[q][3] *= a_hi;
                    }
                const uint32_t vslot = static_cast<uint32_t>(__cvta_generic_to_shared(vring + (i % kVSlots) * vbytes));
                const T* pt = pth;
#pragma unroll
                for (int ks = 0; ks < kStreamTK / 16; ++ks) {
                    uint32_t a[4];
                    a[0] = *reinterpret_cast<const uint32_t*>(&pt[g * kPthPitch + 16 * ks + 2 * cc]);
                    a[1] = *reinterpret_cast<const uint32_t*>(&pt[(g + 8) * kPthPitch + 16 * ks + 2 * cc]);
                    a[2] = *reinterpret_cast<const uint32_t*>(&pt[g * kPthPitch + 16 * ks + 8 + 2 * cc]);
                    a[3] = *reinterpret_cast<const uint32_t*>(&pt[(g + 8) * kPthPitch + 16 * ks + 8 + 2 * cc]);
                    const int vkey = 16 * ks + (mi & 1) * 8 + r8;  // this lane's row address for the V matrices
                    if (ntw == 1) {
                        uint32_t b0, b1;
                        ldsm_x2_t(vslot + 16 * (vkey * uv + swz(vkey, wb, uv)), b0, b1);
                        mma16816<T>(oc[0], a, b0, b1);
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; q += 2)
                            if (q < ntw) {
                                uint32_t b0, b1, b2, b3;
                                const int unit = wb * ntw + q + (mi >> 1);
                                ldsm_x4_t(vslot + 16 * (vkey * uv + swz(vkey, unit, uv)), b0, b1, b2, b3);
                                mma16816<T>(oc[q], a, b0, b1);
                                mma16816<T>(oc[q + 1], a, b2, b3);
                            }
                    }
                }
            }
        }
        // the chunk's partial O, over the rings: every K copy landed before
        // the last scores, every V copy before the last P V
        if (pv_warp) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < ntw) {
                    const int col = 8 * (wb * ntw + q) + 2 * cc;
                    if (g < R) *reinterpret_cast<float2*>(&op[g * Dv + col]) = make_float2(oc[q][0], oc[q][1]);
                    if (g + 8 < R)
                        *reinterpret_cast<float2*>(&op[(g + 8) * Dv + col]) = make_float2(oc[q][2], oc[q][3]);
                }
        }
    }
    __syncthreads();
    if (t < R) {
        st[2 * t] = m_run[t];
        st[2 * t + 1] = l_run[t];
    }

    // ---- every CTA's (max, sum) and partial O are published
    cluster_sync();
    if (t < R) {
        float mc[kMaxCluster], lc[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) {
                mc[c] = ld_peer(peer_addr(&st[2 * t], (uint32_t)c));
                lc[c] = ld_peer(peer_addr(&st[2 * t + 1], (uint32_t)c));
            }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) m = fmaxf(m, mc[c]);
        float l = 0.f;
        if (m != -CUDART_INF_F) {
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c)
                if (c < C && mc[c] != -CUDART_INF_F) l += lc[c] * exp2f(mc[c] - m);
        }
        const float L = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
        lse_s[t] = L;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) fac[t * C + c] = (L == -CUDART_INF_F || mc[c] == -CUDART_INF_F) ? 0.f : exp2f(mc[c] - L);
    }
    __syncthreads();

    // this CTA's slice of the O columns, summed over the cluster
    const int cols = (Dv + C - 1) / C;
    const int c0 = (int)crank * cols, c1 = min(Dv, c0 + cols);
    for (int e = t; e < R * max(0, c1 - c0); e += kThreads) {
        const int r = e / (c1 - c0), d = c0 + e % (c1 - c0);
        float part[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) part[c] = ld_peer(peer_addr(&op[r * Dv + d], (uint32_t)c));
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < C) acc = fmaf(fac[r * C + c], part[c], acc);
        const bool dead = lse_s[r] == -CUDART_INF_F;
        T* orow = static_cast<T*>(p.o) + b * p.so0 + row_h[r] * p.so1 + (long long)row_i[r] * p.so2;
        orow[d] = from_f<T>(dead ? 0.f : acc);
    }
    // P of the chunk
    for (int r = 0; r < R; ++r) {
        const float L = lse_s[r];
        T* prow = static_cast<T*>(p.p) + b * p.sp0 + row_h[r] * p.sp1 + (long long)row_i[r] * p.sp2 + k0;
        for (int j = t; j < n; j += kThreads)
            prow[j] = from_f<T>((L == -CUDART_INF_F) ? 0.f : exp2f(ss[r * p.chunk + j] - L));
    }
    if (crank == 0 && p.lse && t < R) {
        const float L = lse_s[t];
        p.lse[((long long)b * p.Hq + row_h[t]) * p.Sq + row_i[t]] = (L == -CUDART_INF_F) ? L : L * kLn2;
    }
    cluster_sync_relaxed();  // no CTA leaves while a peer may still read its shared memory
}


// ---------------------------------------------------------------------------
// Split-KV kernel for long key sequences (few query rows, many keys).
//
// The same cluster decomposition as decode_kernel (one cluster of C CTAs per
// (batch, key/value head), CTA c owns a contiguous chunk of keys, statistics
// and partial O combined through distributed shared memory), with the parts
// that tie decode_kernel to short chunks taken out:
//   * a thread walks its keys t, t + 256, ... of the chunk, K rows read
//     straight into registers with the next 128-byte batch in flight while the
//     current one is used; the scores of the whole chunk stay in shared memory;
//   * V is not staged whole: 64-key sub-tiles stream through a two-slot ring of
//     asynchronous copies (the first two are issued before the score phase);
//   * P V: a thread owns (key group, pair of O columns) and accumulates all R
//     rows, so every V element is read from shared memory once per CTA;
//   * clusters of up to 16 CTAs (non-portable size, 8 where 16 cannot be
//     scheduled).
// ---------------------------------------------------------------------------
constexpr int kSplitMaxCluster = 16;
constexpr int kSplitTK = 64;                 // keys per V sub-tile
constexpr int kSplitSmemBudget = 220 * 1024;

template <typename T, int RM>
__global__ void __launch_bounds__(kThreads, RM <= 8 ? 2 : 1)
split_kernel(const DecParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float lse_s[kMaxRows];
    __shared__ int row_h[kMaxRows], row_i[kMaxRows];

    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    const uint32_t crank = cluster_rank();
    const int C = (int)(gridDim.x);
    const int b = blockIdx.z, hk = blockIdx.y;
    const int k0 = (int)crank * p.chunk;
    const int n = max(0, min(p.Skv, k0 + p.chunk) - k0);
    const int R = p.rows, D = p.D, Dv = p.Dv;
    constexpr int es = (int)sizeof(T);

    uint8_t* vr = smem + p.off_v;                             // [2][kSplitTK][Dv] V ring (dtype)
    float* qs = reinterpret_cast<float*>(smem + p.off_q);     // [R][D] query rows (fp32)
    float* ss = reinterpret_cast<float*>(smem + p.off_s);     // [R][chunk] scores, then rounded P
    float* part = reinterpret_cast<float*>(smem + p.off_o);   // [G][R][Dv] partial O per key group
    float* st = reinterpret_cast<float*>(smem + p.off_stat);  // [R][2] chunk (max, sum)

    const T* K = static_cast<const T*>(p.k) + b * p.sk0 + hk * p.sk1 + (long long)k0 * p.sk2;
    const T* V = static_cast<const T*>(p.v) + b * p.sv0 + hk * p.sv1 + (long long)k0 * p.sv2;
    const int uv = Dv * es / 16;  // 16-byte units per V row
    const int ntile = (n + kSplitTK - 1) / kSplitTK;
    auto issue_v = [&](int tile) {  // one commit group per call (empty past the last tile)
        if (tile < ntile) {
            const int j0 = tile * kSplitTK, len = min(kSplitTK, n - j0);
            uint8_t* dst = vr + (tile & 1) * kSplitTK * Dv * es;
            for (int u = t; u < len * uv; u += kThreads) {
                const int r = u / uv, c = u % uv;
                cp_async16(dst + 16 * u, reinterpret_cast<const uint8_t*>(V + (long long)(j0 + r) * p.sv2) + 16 * c);
            }
        }
        cp_async_commit();
    };

    // ---- 1. query rows (fp32) and the first two V sub-tiles
    for (int e = t; e < R * D; e += kThreads) {
        const int r = e / D, d = e % D;
        const T* qr = static_cast<const T*>(p.q) + b * p.sq0 + (long long)(hk * p.group + r / p.Sq) * p.sq1 +
                      (long long)(r % p.Sq) * p.sq2;
        qs[e] = to_f(qr[d]);
    }
    if (t < R) {
        row_h[t] = hk * p.group + t / p.Sq;
        row_i[t] = t % p.Sq;
    }
    issue_v(0);
    issue_v(1);
    __syncthreads();

    // ---- 2. scores of this thread's keys; unit u = (key t + 256 * (u / nb),
    // bytes [128 * (u % nb), +128) of its K row)
    {
        const int kbytes = D * es;
        const int nb = (kbytes + 127) / 128;
        const int nk = t < n ? (n - t + kThreads - 1) / kThreads : 0;
        const int nu = nk * nb;
        const uint8_t* kbase = reinterpret_cast<const uint8_t*>(K);
        uint4 cur[8], nxt[8];
        auto load_unit = [&](int u, uint4 (&dst)[8]) {
            const int key = t + kThreads * (u / nb), b0 = 128 * (u % nb);
            const uint8_t* src = kbase + ((long long)key * p.sk2) * es + b0;
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (b0 + 16 * x < kbytes) dst[x] = __ldg(reinterpret_cast<const uint4*>(src + 16 * x));
        };
        if (nu > 0) load_unit(0, cur);
        float acc[RM];
#pragma unroll
        for (int r = 0; r < RM; ++r) acc[r] = 0.f;
        for (int u = 0; u < nu; ++u) {
            if (u + 1 < nu) load_unit(u + 1, nxt);
            const int b0 = 128 * (u % nb);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                if (b0 + 16 * x >= kbytes) break;
                const int d = (b0 + 16 * x) / es;
                if constexpr (es == 4) {
                    const float4 kk = make_float4(__uint_as_float(cur[x].x), __uint_as_float(cur[x].y),
                                                  __uint_as_float(cur[x].z), __uint_as_float(cur[x].w));
#pragma unroll
                    for (int r = 0; r < RM; ++r)
                        if (r < R) {
                            const float4 qq = *reinterpret_cast<const float4*>(&qs[r * D + d]);
                            float a = acc[r];
                            a = fmaf(qq.x, kk.x, a);
                            a = fmaf(qq.y, kk.y, a);
                            a = fmaf(qq.z, kk.z, a);
                            a = fmaf(qq.w, kk.w, a);
                            acc[r] = a;
                        }
                } else {
                    const float2 k01 = unpack2<T>(cur[x].x), k23 = unpack2<T>(cur[x].y);
                    const float2 k45 = unpack2<T>(cur[x].z), k67 = unpack2<T>(cur[x].w);
#pragma unroll
                    for (int r = 0; r < RM; ++r)
                        if (r < R) {
                            const float4 qa = *reinterpret_cast<const float4*>(&qs[r * D + d]);
                            const float4 qb = *reinterpret_cast<const float4*>(&qs[r * D + d + 4]);
                            float a = acc[r];
                            a = fmaf(qa.x, k01.x, a);
                            a = fmaf(qa.y, k01.y, a);
                            a = fmaf(qa.z, k23.x, a);
                            a = fmaf(qa.w, k23.y, a);
                            a = fmaf(qb.x, k45.x, a);
                            a = fmaf(qb.y, k45.y, a);
                            a = fmaf(qb.z, k67.x, a);
                            a = fmaf(qb.w, k67.y, a);
                            acc[r] = a;
                        }
                }
            }
            if (u % nb == nb - 1) {  // this key's dot products are complete
                const int j = t + kThreads * (u / nb), key = k0 + j;
#pragma unroll
                for (int r = 0; r < RM; ++r)
                    if (r < R) {
                        float s = __fmul_rn(acc[r], p.c2);
                        if (p.causal && key > row_i[r]) s = -CUDART_INF_F;
                        if (p.mask_kind != kMaskNone) {
                            const long long off = b * p.sm0 + row_h[r] * p.sm1 + (long long)row_i[r] * p.sm2 + key;
                            if (p.mask_kind == kMaskBool) {
                                if (static_cast<const unsigned char*>(p.mask)[off] == 0) s = -CUDART_INF_F;
                            } else {
                                const float m = p.mask_dtype == kF32 ? static_cast<const float*>(p.mask)[off]
                                                                     : to_f(static_cast<const T*>(p.mask)[off]);
                                s = __fmaf_rn(m, kLog2e, s);
                            }
                        }
                        ss[r * p.chunk + j] = s;
                        acc[r] = 0.f;
                    }
            }
#pragma unroll
            for (int x = 0; x < 8; ++x) cur[x] = nxt[x];
        }
    }
    __syncthreads();

    // per-row (max, sum of exp2) of the chunk: one warp per row
    for (int r = warp; r < R; r += kThreads / 32) {
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

    // ---- 3. the cluster's statistics -> the same lse in every CTA
    cluster_sync();
    if (t < R) {
        float mc[kSplitMaxCluster], lc[kSplitMaxCluster];
#pragma unroll
        for (int c = 0; c < kSplitMaxCluster; ++c)
            if (c < C) {
                mc[c] = ld_peer(peer_addr(&st[2 * t], (uint32_t)c));
                lc[c] = ld_peer(peer_addr(&st[2 * t + 1], (uint32_t)c));
            }
        float m = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < kSplitMaxCluster; ++c)
            if (c < C) m = fmaxf(m, mc[c]);
        float l = 0.f;
        if (m != -CUDART_INF_F) {
#pragma unroll
            for (int c = 0; c < kSplitMaxCluster; ++c)
                if (c < C && mc[c] != -CUDART_INF_F) l += lc[c] * exp2f(mc[c] - m);
        }
        lse_s[t] = (m == -CUDART_INF_F || !(l > 0.f)) ? -CUDART_INF_F : m + log2f(l);
    }
    __syncthreads();

    // ---- 4. per V sub-tile: P (stored, kept rounded), then P V
    const int DP = Dv / 2;                // column pairs (Dv is even)
    const int G = kThreads / DP;          // key groups
    const int kg = t / DP, dp = 2 * (t % DP);
    float a0[RM], a1[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) a0[r] = a1[r] = 0.f;
    for (int tile = 0; tile < ntile; ++tile) {
        const int j0 = tile * kSplitTK, len = min(kSplitTK, n - j0);
        for (int e = t; e < R * len; e += kThreads) {
            const int r = e / len, j = j0 + e % len;
            const float L = lse_s[r];
            const float pr = (L == -CUDART_INF_F) ? 0.f : exp2f(ss[r * p.chunk + j] - L);
            const T pt = from_f<T>(pr);
            T* prow = static_cast<T*>(p.p) + b * p.sp0 + row_h[r] * p.sp1 + (long long)row_i[r] * p.sp2;
            prow[k0 + j] = pt;
            ss[r * p.chunk + j] = to_f(pt);
        }
        cp_async_wait_ring();  // this sub-tile's group is complete (at most the next one is pending)
        __syncthreads();
        if (kg < G) {
            const uint8_t* vt = vr + (tile & 1) * kSplitTK * Dv * es;
            for (int jj = kg; jj < len; jj += G) {
                float2 vv;
                if constexpr (es == 4) vv = *reinterpret_cast<const float2*>(vt + (jj * Dv + dp) * 4);
                else vv = unpack2<T>(*reinterpret_cast<const uint32_t*>(vt + (jj * Dv + dp) * 2));
                const float* pc = ss + j0 + jj;
#pragma unroll
                for (int r = 0; r < RM; ++r)
                    if (r < R) {
                        const float pv = pc[r * p.chunk];
                        a0[r] = fmaf(pv, vv.x, a0[r]);
                        a1[r] = fmaf(pv, vv.y, a1[r]);
                    }
            }
        }
        __syncthreads();   // every thread is done with this ring slot
        issue_v(tile + 2);
    }
    cp_async_wait_all();
    if (kg < G) {
#pragma unroll
        for (int r = 0; r < RM; ++r)
            if (r < R) *reinterpret_cast<float2*>(&part[(kg * R + r) * Dv + dp]) = make_float2(a0[r], a1[r]);
    }
    __syncthreads();
    for (int e = t; e < R * Dv; e += kThreads) {  // sum of the key groups, in place in group 0
        float s = 0.f;
        for (int g = 0; g < G; ++g) s += part[g * R * Dv + e];
        part[e] = s;
    }

    // ---- 5. sum this CTA's slice of the O columns over the cluster
    cluster_sync();
    const int cols = (Dv + C - 1) / C;
    const int c0 = (int)crank * cols, c1 = min(Dv, c0 + cols);
    for (int e = t; e < R * max(0, c1 - c0); e += kThreads) {
        const int r = e / (c1 - c0), d = c0 + e % (c1 - c0);
        float pc[kSplitMaxCluster];
#pragma unroll
        for (int c = 0; c < kSplitMaxCluster; ++c)
            if (c < C) pc[c] = ld_peer(peer_addr(&part[r * Dv + d], (uint32_t)c));
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kSplitMaxCluster; ++c)
            if (c < C) acc += pc[c];
        const bool dead = lse_s[r] == -CUDART_INF_F;
        T* orow = static_cast<T*>(p.o) + b * p.so0 + row_h[r] * p.so1 + (long long)row_i[r] * p.so2;
        orow[d] = from_f<T>(dead ? 0.f : acc);
    }
    if (crank == 0 && p.lse && t < R) {
        const float L = lse_s[t];
        p.lse[((long long)b * p.Hq + row_h[t]) * p.Sq + row_i[t]] = (L == -CUDART_INF_F) ? L : L * kLn2;
    }
    cluster_sync();
}

int elem_bytes(int dt) { return dt == kF32 ? 4 : 2; }

// Cluster size and chunk for a problem, and the shared-memory bytes it needs.
void plan(const Problem& p, int* C, int* chunk, DecParams* dp, int* smem) {
    int c = (int)((p.Skv + 127) / 128);
    c = c < 1 ? 1 : (c > kMaxCluster ? kMaxCluster : c);
    *C = c;
    *chunk = (int)((p.Skv + c - 1) / c);
    const int rows = (int)(p.group * p.Sq);
    int off = 0;
    dp->off_v = off; off += *chunk * (int)p.Dv * elem_bytes(p.dtype); off = (off + 15) & ~15;
    dp->off_q = off; off += rows * (int)p.D * 4; off = (off + 15) & ~15;
    dp->off_s = off; off += rows * *chunk * 4; off = (off + 15) & ~15;
    dp->off_o = off; off += rows * (int)p.Dv * 4; off = (off + 15) & ~15;
    dp->off_stat = off; off += rows * 2 * 4;
    *smem = off;
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

std::mutex g_mu;
struct Ready { const void* kern; int dev; };
Ready g_ready[32];
int g_nready = 0;

void fill_params(const Problem& pr, DecParams* p) {
    p->q = pr.q; p->sq0 = pr.sq[0]; p->sq1 = pr.sq[1]; p->sq2 = pr.sq[2];
    p->k = pr.k; p->sk0 = pr.sk[0]; p->sk1 = pr.sk[1]; p->sk2 = pr.sk[2];
    p->v = pr.v; p->sv0 = pr.sv[0]; p->sv1 = pr.sv[1]; p->sv2 = pr.sv[2];
    p->mask = pr.mask; p->mask_kind = pr.mask_kind; p->mask_dtype = pr.mask_dtype;
    p->sm0 = pr.sm[0]; p->sm1 = pr.sm[1]; p->sm2 = pr.sm[2];
    p->o = pr.o; p->so0 = pr.so[0]; p->so1 = pr.so[1]; p->so2 = pr.so[2];
    p->p = pr.p; p->sp0 = pr.sp[0]; p->sp1 = pr.sp[1]; p->sp2 = pr.sp[2];
    p->lse = pr.lse;
    p->Hq = (int)pr.Hq; p->Sq = (int)pr.Sq; p->Skv = (int)pr.Skv; p->D = (int)pr.D; p->Dv = (int)pr.Dv;
    p->group = (int)pr.group; p->rows = (int)(pr.group * pr.Sq); p->causal = pr.causal;
    p->c2 = pr.scale * kLog2e;
}

template <typename T, int RM>
cudaError_t launch_rm(const Problem& pr, cudaStream_t stream) {
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    int C, chunk, smem;
    plan(pr, &C, &chunk, &p, &smem);
    fill_params(pr, &p);
    p.chunk = chunk;

    auto kern = decode_kernel<T, RM>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        // once per (kernel, device): opt in to the shared-memory budget
        std::lock_guard<std::mutex> lock(g_mu);
        bool ready = false;
        for (int i = 0; i < g_nready; ++i)
            ready |= g_ready[i].kern == reinterpret_cast<const void*>(kern) && g_ready[i].dev == dev;
        if (!ready) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
            if (e != cudaSuccess) return e;
            if (g_nready < 32) g_ready[g_nready++] = Ready{reinterpret_cast<const void*>(kern), dev};
        }
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)C, (unsigned)pr.Hkv, (unsigned)pr.B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Shared-memory layout of stream_decode_kernel: two K and three V slots of
// 32-key pieces (the partial O reuses them after the loop), the chunk's
// scores, two P~ tiles, the k-group partial scores and the merge area.  False
// when it exceeds the budget.
bool plan_stream(const Problem& p, DecParams* dp, int* smem) {
    int C, chunk, smem_cluster;
    DecParams tmp;
    plan(p, &C, &chunk, &tmp, &smem_cluster);
    const long long R = p.group * p.Sq, es = elem_bytes(p.dtype);
    const long long RM = R <= 4 ? 4 : (R <= 8 ? 8 : 16);  // the kernel's row bound
    const long long rings = (long long)kStreamTK * (kKSlots * p.D + kVSlots * p.Dv) * es;
    auto al = [](long long x) { return (x + 15) & ~15ll; };
    long long off = 0;
    const long long off_ring = off; off = al(off + std::max(rings, R * p.Dv * 4));
    const long long off_s = off; off = al(off + R * chunk * 4);
    const long long off_pt = off; off = al(off + 16 * kPthPitch * es);
    const long long off_part = off; off = al(off + 2 * 2 * RM * kStreamTK * 4);
    const long long off_st = off; off = al(off + R * 2 * 4);
    const long long off_fac = off; off += R * C * 4;
    if (off > kSmemBudget) return false;
    dp->off_ring = (int)off_ring;
    dp->off_s = (int)off_s;
    dp->off_pt = (int)off_pt;
    dp->off_part = (int)off_part;
    dp->off_stat = (int)off_st;
    dp->off_fac = (int)off_fac;
    dp->chunk = chunk;
    *smem = (int)off;
    return true;
}

bool pow2_head_dim(int64_t d) { return d == 32 || d == 64 || d == 128 || d == 256; }

// Whether stream_decode_kernel serves p (decode_supports(p) holds already).
bool stream_supports(const Problem& p) {
    if (p.dtype != kF16 && p.dtype != kBF16) return false;
    if (!pow2_head_dim(p.D) || !pow2_head_dim(p.Dv)) return false;
    int smem;
    DecParams dp;
    return plan_stream(p, &dp, &smem);
}

// The register-K cluster kernel stays reachable for 16-bit calls through
// SDPA_MATH_DECODE_KERNEL=cluster.
bool stream_disabled() {
    const char* e = std::getenv("SDPA_MATH_DECODE_KERNEL");
    return e && std::strcmp(e, "cluster") == 0;
}

template <typename T, int RM>
cudaError_t launch_stream_rm(const Problem& pr, cudaStream_t stream) {
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    int smem;
    if (!plan_stream(pr, &p, &smem)) return cudaErrorNotSupported;
    const int chunk = p.chunk;
    fill_params(pr, &p);
    p.chunk = chunk;
    p.k_contig = pr.sk[2] == pr.D;
    p.v_contig = pr.sv[2] == pr.Dv;
    int C, chunk_cluster, smem_cluster;
    {
        DecParams tmp;
        plan(pr, &C, &chunk_cluster, &tmp, &smem_cluster);  // the cluster size plan_stream laid out for
    }

    auto kern = stream_decode_kernel<T, RM>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        bool ready = false;
        for (int i = 0; i < g_nready; ++i)
            ready |= g_ready[i].kern == reinterpret_cast<const void*>(kern) && g_ready[i].dev == dev;
        if (!ready) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
            if (e != cudaSuccess) return e;
            if (g_nready < 32) g_ready[g_nready++] = Ready{reinterpret_cast<const void*>(kern), dev};
        }
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)C, (unsigned)pr.Hkv, (unsigned)pr.B);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_stream_t(const Problem& p, cudaStream_t stream) {
    const int64_t rows = p.group * p.Sq;
    if (rows <= 4) return launch_stream_rm<T, 4>(p, stream);
    if (rows <= 8) return launch_stream_rm<T, 8>(p, stream);
    return launch_stream_rm<T, 16>(p, stream);
}

// Shared-memory layout of split_kernel for a cluster of C CTAs; false when it
// exceeds the budget.
bool plan_split(const Problem& p, int C, int* chunk, DecParams* dp, int* smem) {
    const long long ch = (p.Skv + C - 1) / C;
    const long long rows = p.group * p.Sq, es = elem_bytes(p.dtype);
    const long long G = kThreads / (p.Dv / 2);
    long long off = 0;
    auto al = [](long long x) { return (x + 15) & ~15ll; };
    const long long off_v = off; off = al(off + 2ll * kSplitTK * p.Dv * es);
    const long long off_q = off; off = al(off + rows * p.D * 4);
    const long long off_s = off; off = al(off + rows * ch * 4);
    const long long off_o = off; off = al(off + G * rows * p.Dv * 4);
    const long long off_st = off; off += rows * 2 * 4;
    if (off > kSplitSmemBudget) return false;
    *chunk = (int)ch;
    dp->off_v = (int)off_v; dp->off_q = (int)off_q; dp->off_s = (int)off_s; dp->off_o = (int)off_o;
    dp->off_stat = (int)off_st;
    *smem = (int)off;
    return true;
}

// Cluster size per (kernel, device, shared memory): 16 where the GPU can
// schedule such a cluster with that much shared memory per CTA, else 8.
struct SplitChoice { const void* kern; int dev; int smem; int C; };
SplitChoice g_split[64];
int g_nsplit = 0;
const void* g_split_attr_kern[64];
int g_split_attr_dev[64];
int g_nsplit_attr = 0;

template <typename T, int RM>
cudaError_t launch_split_rm(const Problem& pr, cudaStream_t stream) {
    auto kern = split_kernel<T, RM>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    bool ready = false;
    for (int i = 0; i < g_nsplit_attr; ++i)
        ready |= g_split_attr_kern[i] == reinterpret_cast<const void*>(kern) && g_split_attr_dev[i] == dev;
    if (!ready) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmemBudget);
        if (e != cudaSuccess) return e;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            (void)cudaGetLastError();  // then only portable sizes are offered below
        if (g_nsplit_attr < 64) {
            g_split_attr_kern[g_nsplit_attr] = reinterpret_cast<const void*>(kern);
            g_split_attr_dev[g_nsplit_attr++] = dev;
        }
    }
    DecParams p;
    std::memset(&p, 0, sizeof(p));
    fill_params(pr, &p);
    int chunk = 0, smem = 0, C = kSplitMaxCluster;
    if (!plan_split(pr, C, &chunk, &p, &smem)) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int chosen = 0;
    for (int i = 0; i < g_nsplit; ++i)
        if (g_split[i].kern == reinterpret_cast<const void*>(kern) && g_split[i].dev == dev && g_split[i].smem == smem)
            chosen = g_split[i].C;
    if (chosen == 0) {
        int nc = 0;
        cfg.gridDim = dim3((unsigned)kSplitMaxCluster, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        attr[0].val.clusterDim.x = (unsigned)kSplitMaxCluster;
        if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            nc = 0;
        }
        chosen = nc > 0 ? kSplitMaxCluster : kMaxCluster;
        if (g_nsplit < 64) g_split[g_nsplit++] = SplitChoice{reinterpret_cast<const void*>(kern), dev, smem, chosen};
    }
    C = chosen;
    if (C != kSplitMaxCluster && !plan_split(pr, C, &chunk, &p, &smem)) return cudaErrorNotSupported;
    p.chunk = chunk;
    cfg.gridDim = dim3((unsigned)C, (unsigned)pr.Hkv, (unsigned)pr.B);
    cfg.dynamicSmemBytes = (size_t)smem;
    attr[0].val.clusterDim.x = (unsigned)C;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_split_t(const Problem& p, cudaStream_t stream) {
    const int64_t rows = p.group * p.Sq;
    if (rows <= 4) return launch_split_rm<T, 4>(p, stream);
    if (rows <= 8) return launch_split_rm<T, 8>(p, stream);
    return launch_split_rm<T, 16>(p, stream);
}

template <typename T>
cudaError_t launch_t(const Problem& p, cudaStream_t stream) {
    const int64_t rows = p.group * p.Sq;
    if (rows <= 4) return launch_rm<T, 4>(p, stream);
    if (rows <= 8) return launch_rm<T, 8>(p, stream);
    return launch_rm<T, 16>(p, stream);
}

}  // namespace

bool decode_supports(const Problem& p, const char** why) {
    if (p.group * p.Sq > kMaxRows) { *why = "more than 16 query rows per key/value head"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (p.D > 256 || p.Dv > 256) { *why = "head dim above 256"; return false; }
    if (p.D < 1 || p.Dv < 1) { *why = "empty head dim"; return false; }
    if (p.B > 65535 || p.Hkv > 65535 || p.Skv >= (1ll << 31)) { *why = "sizes beyond the grid limits"; return false; }
    const int es = elem_bytes(p.dtype);
    if ((p.D * es) % 16 != 0 || (p.Dv * es) % 16 != 0) { *why = "head dims must be 16-byte multiples"; return false; }
    if (!aligned16(p.k) || !aligned16(p.v) || (p.sk[2] * es) % 16 != 0 || (p.sv[2] * es) % 16 != 0 ||
        (p.Hkv > 1 && ((p.sk[1] * es) % 16 != 0 || (p.sv[1] * es) % 16 != 0)) ||
        (p.B > 1 && ((p.sk[0] * es) % 16 != 0 || (p.sv[0] * es) % 16 != 0))) {
        *why = "k and v rows must be 16-byte aligned"; return false;
    }
    int C, chunk, smem;
    DecParams dp;
    plan(p, &C, &chunk, &dp, &smem);
    if (chunk > kThreads) { *why = "more than 2048 keys (one thread per key of a chunk)"; return false; }
    if (smem > kSmemBudget) { *why = "key chunk too long for shared memory"; return false; }
    return true;
}

bool split_supports(const Problem& p, const char** why) {
    if (p.group * p.Sq > kMaxRows) { *why = "more than 16 query rows per key/value head"; return false; }
    if (p.Sq < 1 || p.Skv < 1) { *why = "empty sequence"; return false; }
    if (p.D > 256 || p.Dv > 256) { *why = "head dim above 256"; return false; }
    if (p.D < 1 || p.Dv < 1) { *why = "empty head dim"; return false; }
    if (p.B > 65535 || p.Hkv > 65535 || p.Skv >= (1ll << 31)) { *why = "sizes beyond the grid limits"; return false; }
    const int es = elem_bytes(p.dtype);
    if ((p.D * es) % 16 != 0 || (p.Dv * es) % 16 != 0) { *why = "head dims must be 16-byte multiples"; return false; }
    if (!aligned16(p.k) || !aligned16(p.v) || (p.sk[2] * es) % 16 != 0 || (p.sv[2] * es) % 16 != 0 ||
        (p.Hkv > 1 && ((p.sk[1] * es) % 16 != 0 || (p.sv[1] * es) % 16 != 0)) ||
        (p.B > 1 && ((p.sk[0] * es) % 16 != 0 || (p.sv[0] * es) % 16 != 0))) {
        *why = "k and v rows must be 16-byte aligned"; return false;
    }
    int chunk, smem;
    DecParams dp;
    if (!plan_split(p, kSplitMaxCluster, &chunk, &dp, &smem)) {
        *why = "the scores of a 1/16 key chunk do not fit shared memory"; return false;
    }
    return true;
}

cudaError_t launch_split(const Problem& p, cudaStream_t stream) {
    const char* why;
    if (!split_supports(p, &why)) return cudaErrorNotSupported;
    switch (p.dtype) {
        case kF32: return launch_split_t<float>(p, stream);
        case kF16: return launch_split_t<__half>(p, stream);
        case kBF16: return launch_split_t<__nv_bfloat16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const Problem& p, cudaStream_t stream) {
    const char* why;
    if (!decode_supports(p, &why)) return cudaErrorNotSupported;
    if (!stream_disabled() && stream_supports(p))
        return p.dtype == kF16 ? launch_stream_t<__half>(p, stream) : launch_stream_t<__nv_bfloat16>(p, stream);
    switch (p.dtype) {
        case kF32: return launch_t<float>(p, stream);
        case kF16: return launch_t<__half>(p, stream);
        case kBF16: return launch_t<__nv_bfloat16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdpa
