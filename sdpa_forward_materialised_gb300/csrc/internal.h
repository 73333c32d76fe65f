// internal.h -- validated problem descriptor shared by the host API and the
// kernel launchers of the materialised-probability SDPA forward.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sdpa {

enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2, kBool = 3 };
enum MaskKind : int { kMaskNone = 0, kMaskBool = 1, kMaskAdditive = 2 };

// Everything a kernel needs, after host validation.  Strides are in elements;
// a broadcast mask extent has stride 0.  Rows are indexed (b, h, i) with the
// key/value head of query head h equal to h / group.
struct Problem {
    int dtype;  // DType of q, k, v, out, probs
    int64_t B, Hq, Hkv, Sq, Skv, D, Dv, group;
    const void* q;  int64_t sq[4];
    const void* k;  int64_t sk[4];
    const void* v;  int64_t sv[4];
    const void* mask; int mask_kind; int mask_dtype; int64_t sm[4];
    int causal;
    float scale;
    void* o;  int64_t so[4];
    void* p;  int64_t sp[4];
    float* lse;  // optional [B, Hq, Sq] contiguous, natural-log LSE
};

// Number of 128x128 score tiles that survive top-left causal truncation for
// one (b, h) slice.
inline int64_t live_tiles_per_slice(int64_t Sq, int64_t Skv, bool causal) {
    const int64_t tq = (Sq + 127) / 128, tk = (Skv + 127) / 128;
    if (!causal) return tq * tk;
    int64_t n = 0;
    for (int64_t t = 0; t < tq; ++t) {
        const int64_t last_row = (t + 1) * 128 - 1 < Sq - 1 ? (t + 1) * 128 - 1 : Sq - 1;
        const int64_t keys = last_row + 1 < Skv ? last_row + 1 : Skv;
        n += (keys + 127) / 128;
    }
    return n;
}

// Live 128-key tiles of the row block that keeps the most of them (the last
// one) after top-left causal truncation: every row block of a call has at most
// this many key tiles with a visible key.
inline int64_t max_live_key_tiles(int64_t Sq, int64_t Skv, bool causal) {
    if (Sq <= 0 || Skv <= 0) return 0;
    if (!causal) return (Skv + 127) / 128;
    const int64_t last = (Sq - 1 < Skv - 1 ? Sq - 1 : Skv - 1);
    return last / 128 + 1;
}

// The backward's validated arguments (element strides for [B, H, S] of every
// tensor; the innermost stride is 1).  dprobs may be null (no gradient through
// P); rowsum is the caller's B*Hq*Sq float buffer for sum_j P dP per row.
struct BwdProblem {
    int dtype;
    int64_t B, Hq, Hkv, Sq, Skv, D, Dv, group;
    const void* q;  int64_t sq[3];
    const void* k;  int64_t sk[3];
    const void* v;  int64_t sv[3];
    const void* p;  int64_t sp[3];
    const void* dout; int64_t sgo[3];
    const void* dprobs; int64_t sgp[3];
    void* dq; int64_t sdq[3];
    void* dk; int64_t sdk[3];
    void* dv; int64_t sdv[3];
    float* rowsum;
    float scale;
};

// Kernel launchers.  Each returns cudaSuccess or the launch error.  `why`
// receives a static reason string when a launcher cannot serve the problem
// (then it returns cudaErrorNotSupported without launching).
cudaError_t launch_simt(const Problem& p, cudaStream_t stream);
bool tc_supports(const Problem& p, bool fused, const char** why);
// mode 1: two-pass kernel, one 128-row query tile per CTA; 2: two-pass kernel,
// two query tiles per CTA; 3: fused single-sweep kernel; 4: one-sweep cluster kernel.
cudaError_t launch_tc(const Problem& p, int mode, cudaStream_t stream);
bool onesweep_supports(const Problem& p, const char** why);
// Query tiles per CTA that suit the two-pass kernel for p (1 or 2).
int tc_query_tiles(const Problem& p);
// Whether AUTO serves p with the one-sweep cluster kernel.
bool onesweep_auto(const Problem& p);
bool decode_supports(const Problem& p, const char** why);
cudaError_t launch_decode(const Problem& p, cudaStream_t stream);
bool split_supports(const Problem& p, const char** why);
bool tc_decode_supports(const Problem& p, const char** why);
cudaError_t launch_tc_decode(const Problem& p, cudaStream_t stream);
cudaError_t launch_split(const Problem& p, cudaStream_t stream);
cudaError_t launch_bwd(const BwdProblem& p, cudaStream_t stream);   // CUDA-core kernels, any shape
bool bwd_tc_supports(const BwdProblem& p, const char** why);
cudaError_t launch_bwd_tc(const BwdProblem& p, cudaStream_t stream);  // tensor-core kernels

// Device error word shared by every kernel of the library (see
// sdpa_math_device_status).  read_and_clear returns the word's old value.
cudaError_t status_read_and_clear(cudaStream_t stream, unsigned int* value);
// Enqueue the bounded-wait self test (see sdpa_math_selftest_wait).
cudaError_t launch_selftest_wait(cudaStream_t stream);

}  // namespace sdpa
