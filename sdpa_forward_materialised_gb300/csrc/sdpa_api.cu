// sdpa_api.cu -- host side of the C ABI declared in include/sdpa_math.h:
// argument validation (before any launch), kernel-family selection by counted
// live score tiles, and dispatch to the launchers.
//
// Semantics enforced here follow FlagOS-OP PR #10 "feat: add sdpa_math
// operator" (overview, "semantics" item): causal and attn_mask are mutually
// exclusive, GQA needs Hq % Hkv == 0, dropout is not part of the call; the
// "_d1()" micro-optimisation item (2026-10-02 update) fixes the layout rule
// that only the innermost stride must be 1.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <mutex>

#include "sdpa_math.h"  // include/ is on the compiler search path
#include "internal.h"

namespace {

thread_local std::string g_last_error;

sdpa_status fail(sdpa_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

// SDPA_MATH_VARIANT=auto|simt|twopass|paired|fused|decode|split|tcdecode, read once at load.
sdpa_variant env_variant() {
    static const sdpa_variant v = [] {
        const char* e = std::getenv("SDPA_MATH_VARIANT");
        if (!e || !*e || !std::strcmp(e, "auto")) return SDPA_VARIANT_AUTO;
        if (!std::strcmp(e, "simt")) return SDPA_VARIANT_SIMT;
        if (!std::strcmp(e, "twopass")) return SDPA_VARIANT_TC_TWOPASS;
        if (!std::strcmp(e, "paired")) return SDPA_VARIANT_TC_PAIRED;
        if (!std::strcmp(e, "fused")) return SDPA_VARIANT_TC_FUSED;
        if (!std::strcmp(e, "decode")) return SDPA_VARIANT_DECODE;
        if (!std::strcmp(e, "split")) return SDPA_VARIANT_SPLIT;
        if (!std::strcmp(e, "tcdecode")) return SDPA_VARIANT_TC_DECODE;
        if (!std::strcmp(e, "onesweep")) return SDPA_VARIANT_TC_ONESWEEP;
        return SDPA_VARIANT_AUTO;
    }();
    return v;
}

int64_t elem_size(int dt) {
    switch (dt) {
        case SDPA_F32: return 4;
        case SDPA_F16: case SDPA_BF16: return 2;
        case SDPA_BOOL: return 1;
        default: return 0;
    }
}

const char* dtype_name(int dt) {
    switch (dt) {
        case SDPA_F32: return "f32";
        case SDPA_F16: return "f16";
        case SDPA_BF16: return "bf16";
        case SDPA_BOOL: return "bool";
        default: return "unknown";
    }
}

int64_t numel(const sdpa_tensor* t) {
    int64_t n = 1;
    for (int i = 0; i < 4; ++i) n *= t->shape[i];
    return n;
}

// Checks shared by every tensor argument.
sdpa_status check_tensor(const sdpa_tensor* t, const char* name) {
    if (!t) return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: tensor descriptor is NULL", name);
    for (int i = 0; i < 4; ++i) {
        if (t->shape[i] < 0)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: negative extent shape[%d]=%lld", name, i,
                        (long long)t->shape[i]);
        if (t->stride[i] < 0)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: negative stride[%d]", name, i);
    }
    const int64_t es = elem_size(t->dtype);
    if (es == 0) return fail(SDPA_ERR_UNSUPPORTED, "%s: unknown dtype %d", name, (int)t->dtype);
    if (numel(t) > 0) {
        if (!t->data) return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: data pointer is NULL", name);
        if (((uintptr_t)t->data) % (uintptr_t)es != 0)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: data pointer not aligned to its %lld-byte element",
                        name, (long long)es);
        if (t->shape[3] > 1 && t->stride[3] != 1)
            return fail(SDPA_ERR_INVALID_ARGUMENT,
                        "%s: innermost stride must be 1 (got %lld)", name, (long long)t->stride[3]);
    }
    return SDPA_OK;
}

// An output must not overlap itself: no dimension of extent > 1 may have
// stride 0 (a broadcast view), or its elements would be written by several
// threads at once.
sdpa_status check_output(const sdpa_tensor* t, const char* name) {
    for (int i = 0; i < 4; ++i)
        if (t->shape[i] > 1 && t->stride[i] == 0)
            return fail(SDPA_ERR_INVALID_ARGUMENT,
                        "%s: dimension %d has stride 0 over %lld elements (an output must not overlap itself)",
                        name, i, (long long)t->shape[i]);
    return SDPA_OK;
}

bool same_shape(const sdpa_tensor* t, int64_t a, int64_t b, int64_t c, int64_t d) {
    return t->shape[0] == a && t->shape[1] == b && t->shape[2] == c && t->shape[3] == d;
}

// Full validation; fills `p` on success.
sdpa_status validate(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                     const sdpa_tensor* mask, sdpa_mask_kind mask_kind, int is_causal, float scale,
                     const sdpa_tensor* out, const sdpa_tensor* probs, sdpa::Problem* p) {
    sdpa_status s;
    if ((s = check_tensor(q, "q")) != SDPA_OK) return s;
    if ((s = check_tensor(k, "k")) != SDPA_OK) return s;
    if ((s = check_tensor(v, "v")) != SDPA_OK) return s;
    if ((s = check_tensor(out, "out")) != SDPA_OK) return s;
    if ((s = check_tensor(probs, "probs")) != SDPA_OK) return s;
    if ((s = check_output(out, "out")) != SDPA_OK) return s;
    if ((s = check_output(probs, "probs")) != SDPA_OK) return s;

    if (q->dtype != SDPA_F32 && q->dtype != SDPA_F16 && q->dtype != SDPA_BF16)
        return fail(SDPA_ERR_UNSUPPORTED, "q: dtype %s is not f32/f16/bf16", dtype_name(q->dtype));
    const sdpa_tensor* same[] = {k, v, out, probs};
    const char* names[] = {"k", "v", "out", "probs"};
    for (int i = 0; i < 4; ++i)
        if (same[i]->dtype != q->dtype)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: dtype %s differs from q dtype %s", names[i],
                        dtype_name(same[i]->dtype), dtype_name(q->dtype));

    const int64_t B = q->shape[0], Hq = q->shape[1], Sq = q->shape[2], D = q->shape[3];
    const int64_t Hkv = k->shape[1], Skv = k->shape[2], Dv = v->shape[3];
    if (k->shape[0] != B || v->shape[0] != B)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "batch mismatch: q %lld, k %lld, v %lld", (long long)B,
                    (long long)k->shape[0], (long long)v->shape[0]);
    if (v->shape[1] != Hkv)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "k and v disagree on heads (%lld vs %lld)",
                    (long long)Hkv, (long long)v->shape[1]);
    if (v->shape[2] != Skv)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "k and v disagree on key length (%lld vs %lld)",
                    (long long)Skv, (long long)v->shape[2]);
    if (k->shape[3] != D)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "q and k disagree on head dim (%lld vs %lld)",
                    (long long)D, (long long)k->shape[3]);
    if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0)
        return fail(SDPA_ERR_INVALID_ARGUMENT,
                    "GQA requires Hq divisible by Hkv (Hq=%lld, Hkv=%lld)", (long long)Hq,
                    (long long)Hkv);
    if (is_causal && mask_kind != SDPA_MASK_NONE)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "is_causal and an attention mask are mutually exclusive");
    if (!std::isfinite(scale)) return fail(SDPA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (D > 256 || Dv > 256)
        return fail(SDPA_ERR_UNSUPPORTED, "head dim above 256 is not supported (D=%lld, Dv=%lld)",
                    (long long)D, (long long)Dv);
    if (!same_shape(out, B, Hq, Sq, Dv))
        return fail(SDPA_ERR_INVALID_ARGUMENT, "out must be [B,Hq,Sq,Dv] = [%lld,%lld,%lld,%lld]",
                    (long long)B, (long long)Hq, (long long)Sq, (long long)Dv);
    if (!same_shape(probs, B, Hq, Sq, Skv))
        return fail(SDPA_ERR_INVALID_ARGUMENT, "probs must be [B,Hq,Sq,Skv] = [%lld,%lld,%lld,%lld]",
                    (long long)B, (long long)Hq, (long long)Sq, (long long)Skv);

    std::memset(p, 0, sizeof(*p));
    if (mask_kind == SDPA_MASK_NONE) {
        if (mask) return fail(SDPA_ERR_INVALID_ARGUMENT, "mask given with mask_kind NONE");
    } else if (mask_kind == SDPA_MASK_BOOL || mask_kind == SDPA_MASK_ADDITIVE) {
        if (!mask) return fail(SDPA_ERR_INVALID_ARGUMENT, "mask_kind set but mask is NULL");
        if ((s = check_tensor(mask, "mask")) != SDPA_OK) return s;
        const int64_t mb = mask->shape[0], mh = mask->shape[1];
        if (!(mb == 1 || mb == B) || !(mh == 1 || mh == Hq) || mask->shape[2] != Sq ||
            mask->shape[3] != Skv)
            return fail(SDPA_ERR_INVALID_ARGUMENT,
                        "mask shape must be [1|B, 1|Hq, Sq, Skv] = [1|%lld, 1|%lld, %lld, %lld]",
                        (long long)B, (long long)Hq, (long long)Sq, (long long)Skv);
        if (mask_kind == SDPA_MASK_BOOL && mask->dtype != SDPA_BOOL)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "a bool mask must have dtype bool");
        if (mask_kind == SDPA_MASK_ADDITIVE && mask->dtype != q->dtype && mask->dtype != SDPA_F32)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "an additive mask must have the q dtype or f32");
        p->mask = mask->data;
        p->mask_kind = mask_kind;
        p->mask_dtype = mask->dtype;
        p->sm[0] = (mb == 1) ? 0 : mask->stride[0];
        p->sm[1] = (mh == 1) ? 0 : mask->stride[1];
        p->sm[2] = mask->stride[2];
        p->sm[3] = 1;
    } else {
        return fail(SDPA_ERR_INVALID_ARGUMENT, "unknown mask_kind %d", (int)mask_kind);
    }

    p->dtype = q->dtype;
    p->B = B; p->Hq = Hq; p->Hkv = Hkv; p->Sq = Sq; p->Skv = Skv; p->D = D; p->Dv = Dv;
    p->group = Hkv > 0 ? Hq / Hkv : 1;
    p->q = q->data; p->k = k->data; p->v = v->data; p->o = out->data; p->p = probs->data;
    for (int i = 0; i < 4; ++i) {
        p->sq[i] = q->stride[i]; p->sk[i] = k->stride[i]; p->sv[i] = v->stride[i];
        p->so[i] = out->stride[i]; p->sp[i] = probs->stride[i];
    }
    p->sq[3] = p->sk[3] = p->sv[3] = p->so[3] = p->sp[3] = 1;
    p->causal = is_causal ? 1 : 0;
    p->scale = scale;
    p->lse = nullptr;
    return SDPA_OK;
}

// The single-sweep fused tensor-core kernel keeps the scores of a row block
// in TMEM beside O: at most two live 128-key tiles per row block.
constexpr int64_t kFusedMaxLiveTiles = 2;

// Variant the AUTO rule picks for a validated problem.  The tensor-core
// families are ordered by measurement on GB300 (a sweep over live-tile counts
// 1..16 per row block and 4..16384 tiles per call): the two-pass kernels were
// faster than the fused one at every shape both could run, so the fused
// kernel serves the calls whose rows TMA cannot describe (P rows that are not
// 16-byte multiples) when each row block keeps at most two live key tiles;
// the one-sweep cluster kernel takes causal calls whose clusters all fit in
// one wave (onesweep_auto); between the two two-pass layouts the paired grid
// is taken once it still fills about three quarters of the SMs
// (tc_query_tiles).
sdpa_variant choose(const sdpa::Problem& p) {
    const char* why = nullptr;
    if (p.dtype == SDPA_F32) return SDPA_VARIANT_SIMT;
    if (sdpa::decode_supports(p, &why)) return SDPA_VARIANT_DECODE;
    if (sdpa::tc_decode_supports(p, &why)) return SDPA_VARIANT_TC_DECODE;
    if (sdpa::split_supports(p, &why)) return SDPA_VARIANT_SPLIT;
    if (sdpa::tc_supports(p, false, &why)) {
        if (sdpa::onesweep_auto(p) && sdpa::onesweep_supports(p, &why)) return SDPA_VARIANT_TC_ONESWEEP;
        return sdpa::tc_query_tiles(p) == 2 ? SDPA_VARIANT_TC_PAIRED : SDPA_VARIANT_TC_TWOPASS;
    }
    if (sdpa::max_live_key_tiles(p.Sq, p.Skv, p.causal != 0) <= kFusedMaxLiveTiles && sdpa::tc_supports(p, true, &why))
        return SDPA_VARIANT_TC_FUSED;
    return SDPA_VARIANT_SIMT;
}

sdpa_status resolve(const sdpa::Problem& p, sdpa_variant requested, sdpa_variant* out) {
    sdpa_variant v = requested == SDPA_VARIANT_AUTO ? env_variant() : requested;
    const char* why = "not supported";
    switch (v) {
        case SDPA_VARIANT_AUTO: *out = choose(p); return SDPA_OK;
        case SDPA_VARIANT_SIMT: *out = v; return SDPA_OK;
        case SDPA_VARIANT_TC_TWOPASS:
        case SDPA_VARIANT_TC_PAIRED:
        case SDPA_VARIANT_TC_FUSED:
            if (!sdpa::tc_supports(p, v == SDPA_VARIANT_TC_FUSED, &why))
                return fail(SDPA_ERR_UNSUPPORTED, "tensor-core variant cannot serve this call: %s", why);
            *out = v;
            return SDPA_OK;
        case SDPA_VARIANT_DECODE:
            if (!sdpa::decode_supports(p, &why))
                return fail(SDPA_ERR_UNSUPPORTED, "decode variant cannot serve this call: %s", why);
            *out = v;
            return SDPA_OK;
        case SDPA_VARIANT_SPLIT:
            if (!sdpa::split_supports(p, &why))
                return fail(SDPA_ERR_UNSUPPORTED, "split variant cannot serve this call: %s", why);
            *out = v;
            return SDPA_OK;
        case SDPA_VARIANT_TC_ONESWEEP:
            if (!sdpa::onesweep_supports(p, &why))
                return fail(SDPA_ERR_UNSUPPORTED, "one-sweep variant cannot serve this call: %s", why);
            *out = v;
            return SDPA_OK;
        case SDPA_VARIANT_TC_DECODE:
            if (!sdpa::tc_decode_supports(p, &why))
                return fail(SDPA_ERR_UNSUPPORTED, "tensor-core decode variant cannot serve this call: %s", why);
            *out = v;
            return SDPA_OK;
        default:
            return fail(SDPA_ERR_INVALID_ARGUMENT, "unknown variant %d", (int)v);
    }
}

}  // namespace

extern "C" {

const char* sdpa_math_last_error(void) { return g_last_error.c_str(); }

int sdpa_math_abi_version(void) { return SDPA_MATH_ABI_VERSION; }

sdpa_status sdpa_math_plan(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                           const sdpa_tensor* mask, sdpa_mask_kind mask_kind, int is_causal,
                           float scale, const sdpa_tensor* out, const sdpa_tensor* probs,
                           sdpa_variant requested, sdpa_plan* plan) {
    g_last_error.clear();
    if (!plan) return fail(SDPA_ERR_INVALID_ARGUMENT, "plan is NULL");
    sdpa::Problem p;
    sdpa_status s = validate(q, k, v, mask, mask_kind, is_causal, scale, out, probs, &p);
    if (s != SDPA_OK) return s;
    sdpa_variant chosen;
    if ((s = resolve(p, requested, &chosen)) != SDPA_OK) return s;
    plan->variant = chosen;
    plan->live_score_tiles = p.B * p.Hq * sdpa::live_tiles_per_slice(p.Sq, p.Skv, p.causal != 0);
    plan->launches = (p.B * p.Hq * p.Sq == 0) ? 0 : 1;
    return SDPA_OK;
}

sdpa_status sdpa_math_fwd_ex(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                             const sdpa_tensor* mask, sdpa_mask_kind mask_kind, int is_causal,
                             float scale, sdpa_tensor* out, sdpa_tensor* probs, float* lse,
                             sdpa_variant variant, sdpa_stream_t stream) {
    g_last_error.clear();
    sdpa::Problem p;
    sdpa_status s = validate(q, k, v, mask, mask_kind, is_causal, scale, out, probs, &p);
    if (s != SDPA_OK) return s;
    if (lse && ((uintptr_t)lse) % 4 != 0)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "lse pointer not 4-byte aligned");
    p.lse = lse;
    sdpa_variant chosen;
    if ((s = resolve(p, variant, &chosen)) != SDPA_OK) return s;
    if (p.B * p.Hq * p.Sq == 0) return SDPA_OK;  // nothing to write

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (chosen) {
        case SDPA_VARIANT_TC_TWOPASS: e = sdpa::launch_tc(p, 1, st); break;
        case SDPA_VARIANT_TC_PAIRED: e = sdpa::launch_tc(p, 2, st); break;
        case SDPA_VARIANT_TC_FUSED: e = sdpa::launch_tc(p, 3, st); break;
        case SDPA_VARIANT_TC_ONESWEEP: e = sdpa::launch_tc(p, 4, st); break;
        case SDPA_VARIANT_DECODE: e = sdpa::launch_decode(p, st); break;
        case SDPA_VARIANT_SPLIT: e = sdpa::launch_split(p, st); break;
        case SDPA_VARIANT_TC_DECODE: e = sdpa::launch_tc_decode(p, st); break;
        default: e = sdpa::launch_simt(p, st); break;
    }
    // A family can still refuse at launch, before enqueuing anything: the
    // driver will not encode a TMA descriptor for this layout, or (TC_DECODE)
    // only the portable 8-CTA cluster can be scheduled and a key chunk of that
    // cluster does not fit shared memory.  AUTO then serves the call with the
    // split-KV kernel where it can, else the CUDA-core kernel; a forced family
    // reports it.
    if (e == cudaErrorNotSupported && chosen != SDPA_VARIANT_SIMT) {
        (void)cudaGetLastError();
        if (variant != SDPA_VARIANT_AUTO || env_variant() != SDPA_VARIANT_AUTO)
            return fail(SDPA_ERR_UNSUPPORTED,
                        "the forced kernel family refused its launch: the driver would not encode a TMA "
                        "descriptor for this layout, or the cluster size that can be scheduled leaves a key "
                        "chunk too large for shared memory");
        const char* why = nullptr;
        if (chosen == SDPA_VARIANT_TC_DECODE && sdpa::split_supports(p, &why)) e = sdpa::launch_split(p, st);
        else if (chosen == SDPA_VARIANT_TC_ONESWEEP) e = sdpa::launch_tc(p, 1, st);
        else e = sdpa::launch_simt(p, st);
        if (e == cudaErrorNotSupported) {
            (void)cudaGetLastError();
            e = sdpa::launch_simt(p, st);
        }
    }
    if (e != cudaSuccess)
        return fail(SDPA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return SDPA_OK;
}

sdpa_status sdpa_math_fwd(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                          const sdpa_tensor* mask, sdpa_mask_kind mask_kind, int is_causal,
                          float scale, sdpa_tensor* out, sdpa_tensor* probs, sdpa_stream_t stream) {
    return sdpa_math_fwd_ex(q, k, v, mask, mask_kind, is_causal, scale, out, probs, nullptr,
                            SDPA_VARIANT_AUTO, stream);
}

sdpa_status sdpa_math_device_status(sdpa_stream_t stream) {
    g_last_error.clear();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "stream synchronize failed: %s", cudaGetErrorString(e));
    unsigned int word = 0;
    e = sdpa::status_read_and_clear(st, &word);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "reading the device status failed: %s", cudaGetErrorString(e));
    if (word != 0)
        return fail(SDPA_ERR_TIMEOUT,
                    "a device-side wait ran out of iterations (role %u, barrier %u, block %u)",
                    (word >> 24) & 0xff, (word >> 16) & 0xff, word & 0xffff);
    return SDPA_OK;
}

sdpa_status sdpa_math_bwd_ex(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                             const sdpa_tensor* probs, const sdpa_tensor* dout, const sdpa_tensor* dprobs,
                             float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv, float* rowsum,
                             sdpa_variant variant, sdpa_stream_t stream) {
    g_last_error.clear();
    if (variant != SDPA_VARIANT_AUTO && variant != SDPA_VARIANT_SIMT && variant != SDPA_VARIANT_TC_TWOPASS)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "backward variant must be AUTO, SIMT or TC_TWOPASS (got %d)",
                    (int)variant);
    sdpa_status s;
    const sdpa_tensor* all[] = {q, k, v, probs, dout, dq, dk, dv};
    const char* names[] = {"q", "k", "v", "probs", "dout", "dq", "dk", "dv"};
    for (int i = 0; i < 8; ++i)
        if ((s = check_tensor(all[i], names[i])) != SDPA_OK) return s;
    for (int i = 5; i < 8; ++i)
        if ((s = check_output(all[i], names[i])) != SDPA_OK) return s;
    if (dprobs && (s = check_tensor(dprobs, "dprobs")) != SDPA_OK) return s;
    if (q->dtype != SDPA_F32 && q->dtype != SDPA_F16 && q->dtype != SDPA_BF16)
        return fail(SDPA_ERR_UNSUPPORTED, "q: dtype %s is not f32/f16/bf16", dtype_name(q->dtype));
    for (int i = 1; i < 8; ++i)
        if (all[i]->dtype != q->dtype)
            return fail(SDPA_ERR_INVALID_ARGUMENT, "%s: dtype %s differs from q dtype %s", names[i],
                        dtype_name(all[i]->dtype), dtype_name(q->dtype));
    if (dprobs && dprobs->dtype != q->dtype)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "dprobs: dtype differs from q");
    const int64_t B = q->shape[0], Hq = q->shape[1], Sq = q->shape[2], D = q->shape[3];
    const int64_t Hkv = k->shape[1], Skv = k->shape[2], Dv = v->shape[3];
    if (k->shape[0] != B || !same_shape(v, B, Hkv, Skv, Dv) || k->shape[3] != D)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "k must be [B,Hkv,Skv,D] and v [B,Hkv,Skv,Dv] for q [B,Hq,Sq,D]");
    if (Hkv <= 0 ? Hq != 0 : (Hq % Hkv) != 0)
        return fail(SDPA_ERR_INVALID_ARGUMENT, "GQA requires Hq divisible by Hkv (Hq=%lld, Hkv=%lld)",
                    (long long)Hq, (long long)Hkv);
    if (D > 256 || Dv > 256) return fail(SDPA_ERR_UNSUPPORTED, "head dim above 256 is not supported");
    if (!std::isfinite(scale)) return fail(SDPA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!same_shape(probs, B, Hq, Sq, Skv) || (dprobs && !same_shape(dprobs, B, Hq, Sq, Skv)))
        return fail(SDPA_ERR_INVALID_ARGUMENT, "probs and dprobs must be [B,Hq,Sq,Skv]");
    if (!same_shape(dout, B, Hq, Sq, Dv)) return fail(SDPA_ERR_INVALID_ARGUMENT, "dout must be [B,Hq,Sq,Dv]");
    if (!same_shape(dq, B, Hq, Sq, D) || !same_shape(dk, B, Hkv, Skv, D) || !same_shape(dv, B, Hkv, Skv, Dv))
        return fail(SDPA_ERR_INVALID_ARGUMENT, "dq, dk, dv must have the shapes of q, k, v");
    if (B * Hq * Sq > 0 && (!rowsum || ((uintptr_t)rowsum) % 4 != 0))
        return fail(SDPA_ERR_INVALID_ARGUMENT, "rowsum must be a 4-byte aligned device buffer of B*Hq*Sq floats");
    sdpa::BwdProblem p;
    std::memset(&p, 0, sizeof(p));
    p.dtype = q->dtype;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Sq = Sq; p.Skv = Skv; p.D = D; p.Dv = Dv;
    p.group = Hkv > 0 ? Hq / Hkv : 1;
    auto set = [](const sdpa_tensor* t, const void** ptr, int64_t* st) {
        *ptr = t ? t->data : nullptr;
        for (int i = 0; i < 3; ++i) st[i] = t ? t->stride[i] : 0;
    };
    set(q, &p.q, p.sq); set(k, &p.k, p.sk); set(v, &p.v, p.sv); set(probs, &p.p, p.sp);
    set(dout, &p.dout, p.sgo); set(dprobs, &p.dprobs, p.sgp);
    const void* tmp;
    set(dq, &tmp, p.sdq); p.dq = dq->data;
    set(dk, &tmp, p.sdk); p.dk = dk->data;
    set(dv, &tmp, p.sdv); p.dv = dv->data;
    p.rowsum = rowsum;
    p.scale = scale;
    const char* why = nullptr;
    const bool tc_ok = sdpa::bwd_tc_supports(p, &why);
    if (variant == SDPA_VARIANT_TC_TWOPASS && !tc_ok)
        return fail(SDPA_ERR_UNSUPPORTED, "tensor-core backward cannot serve this call: %s", why);
    if (B * Hkv == 0 || (Sq == 0 && Skv == 0)) return SDPA_OK;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool use_tc = variant == SDPA_VARIANT_TC_TWOPASS || (variant == SDPA_VARIANT_AUTO && tc_ok);
    cudaError_t e = use_tc ? sdpa::launch_bwd_tc(p, st) : sdpa::launch_bwd(p, st);
    if (e == cudaErrorNotSupported && use_tc) {
        (void)cudaGetLastError();
        if (variant != SDPA_VARIANT_AUTO)
            return fail(SDPA_ERR_UNSUPPORTED, "tensor-core backward refused its launch configuration");
        e = sdpa::launch_bwd(p, st);
    }
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return SDPA_OK;
}

sdpa_status sdpa_math_bwd(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                          const sdpa_tensor* probs, const sdpa_tensor* dout, const sdpa_tensor* dprobs,
                          float scale, sdpa_tensor* dq, sdpa_tensor* dk, sdpa_tensor* dv, float* rowsum,
                          sdpa_stream_t stream) {
    return sdpa_math_bwd_ex(q, k, v, probs, dout, dprobs, scale, dq, dk, dv, rowsum, SDPA_VARIANT_AUTO, stream);
}

sdpa_status sdpa_math_selftest_wait(sdpa_stream_t stream) {
    g_last_error.clear();
    const cudaError_t e = sdpa::launch_selftest_wait(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "self-test launch failed: %s", cudaGetErrorString(e));
    return SDPA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- backward without caller scratch
// sdpa_math_bwd takes a caller-allocated B*Hq*Sq float buffer for the per-row
// sums its rows kernel writes and its keys kernel reads.  Callers that cannot
// allocate device memory at call time (a framework that owns all device
// memory through its own pre-planned pool, a real-time path that forbids
// cudaMalloc after start-up) use sdpa_math_bwd_noalloc, which keeps those
// sums in the fixed array below instead.  It lives in the library's own
// device memory on every GPU that loads the library, until the process exits.
// Every call shares it; nothing in it must start at zero, because each call's
// rows kernel writes every row before its keys kernel reads it.  Calls that
// overlap on the GPU race on it.
namespace {

static __device__ __align__(256) float g_bwd_rowsum_scratch[SDPA_BWD_NOALLOC_MAX_ROWS];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices];  // device address of the array, per device (null until looked up)

// Device address of the array on the current device.  In host code the
// array's name is a host-side stand-in, not a device address, so it is looked
// up once per device with that device current and cached.
cudaError_t scratch_address(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_rowsum_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" sdpa_status sdpa_math_bwd_noalloc(const sdpa_tensor* q, const sdpa_tensor* k, const sdpa_tensor* v,
                                             const sdpa_tensor* probs, const sdpa_tensor* dout,
                                             const sdpa_tensor* dprobs, float scale, sdpa_tensor* dq,
                                             sdpa_tensor* dk, sdpa_tensor* dv, sdpa_stream_t stream) {
    g_last_error.clear();
    sdpa_status s = check_tensor(q, "q");
    if (s != SDPA_OK) return s;
    const int64_t rows = q->shape[0] * q->shape[1] * q->shape[2];
    if (rows > (int64_t)SDPA_BWD_NOALLOC_MAX_ROWS)
        return fail(SDPA_ERR_UNSUPPORTED,
                    "sdpa_math_bwd_noalloc serves at most %lld query rows (B*Hq*Sq), got %lld; "
                    "use sdpa_math_bwd with a caller buffer",
                    (long long)SDPA_BWD_NOALLOC_MAX_ROWS, (long long)rows);
    float* rowsum = nullptr;
    const cudaError_t e = scratch_address(&rowsum);
    if (e != cudaSuccess)
        return fail(SDPA_ERR_CUDA, "looking up the library's row-sum array failed: %s", cudaGetErrorString(e));
    return sdpa_math_bwd_ex(q, k, v, probs, dout, dprobs, scale, dq, dk, dv, rowsum, SDPA_VARIANT_AUTO, stream);
}
