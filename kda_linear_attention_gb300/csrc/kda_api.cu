// C-ABI shim of libkda_gb300: argument validation and kernel dispatch.
// Declarations and the contract of each call are in include/kda.h.
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr int kVersion = 200;   // 0.2.0: caller-owned prefill workspace

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

extern "C" {

int kda_version(void) { return kVersion; }

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_DIM: return "unsupported or inconsistent sizes (dk = dv = 128, N >= 1, H >= 1)";
        case KDA_ERR_CHUNK: return "chunk must be 16, 32 or 64";
        case KDA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case KDA_ERR_DTYPE: return "dtype must be KDA_BF16 or KDA_F32";
        case KDA_ERR_WORKSPACE: return "workspace could not be allocated or is too small";
        case KDA_ERR_CUDA: return "CUDA launch error";
        case KDA_ERR_VALUE: return "a scalar argument is out of range (eps >= 0, finite q_scale)";
        default: return "unknown status";
    }
}

int kda_prefill_chunked(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *S0, float *o, float *S_out,
                        const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                        int chunk, int dtype, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_CHUNK;
    if (!S_out || !cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S0, o, S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16 && chunk == 64 && T > 0) {
        const cudaError_t e = kda::launch_prefill_split(q, k, v, g, beta, S0, o, S_out, cu_seqlens,
                                                        N, T, H, s);
        return e == cudaErrorMemoryAllocation ? KDA_ERR_WORKSPACE : cuda_status(e);
    }
    return cuda_status(kda::launch_prefill_simt(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H,
                                                chunk, dtype == KDA_BF16, s));
}

int kda_prefill_chunked_events(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, const float *S0, float *o, float *S_out,
                               const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                               int chunk, int dtype, void *stream, void *const *events) {
    if (!events || !events[0] || !events[1] || !events[2] || !events[3]) return KDA_ERR_NULL;
    if (dtype != KDA_BF16 || chunk != 64 || T <= 0) return KDA_ERR_CHUNK;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (!S_out || !cu_seqlens || !q || !k || !v || !g || !beta || !o) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S0, o, S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) ev[i] = static_cast<cudaEvent_t>(events[i]);
    const cudaError_t e = kda::launch_prefill_split(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N,
                                                    T, H, static_cast<cudaStream_t>(stream), ev);
    return e == cudaErrorMemoryAllocation ? KDA_ERR_WORKSPACE : cuda_status(e);
}

int kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, const float *S0, float *o, float *S_out,
                                const int32_t *cu_seqlens, int N, int64_t T, int H, int dk,
                                int dv, int chunk, int dtype, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_CHUNK;
    if (!S_out || !cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S0, o, S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16 && chunk == 64 && T > 0) {
        if (kda::prefill_split_workspace_bytes(N, T, H) > kda::kNoAllocScratchBytes)
            return KDA_ERR_WORKSPACE;
        return cuda_status(kda::launch_prefill_split_noalloc(q, k, v, g, beta, S0, o, S_out,
                                                             cu_seqlens, N, T, H, s));
    }
    // the CUDA-core kernel needs no workspace
    return cuda_status(kda::launch_prefill_simt(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H,
                                                chunk, dtype == KDA_BF16, s));
}

size_t kda_prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk, int dtype) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return 0;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T <= 0 || T >= (int64_t(1) << 31))
        return 0;
    if (dtype != KDA_BF16 || chunk != 64) return 0;
    return kda::prefill_split_workspace_bytes(N, T, H);
}

int kda_prefill_chunked_ws(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const float *S0, float *o, float *S_out,
                           const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                           int chunk, int dtype, void *workspace, size_t ws_bytes, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_CHUNK;
    if (!S_out || !cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S0, o, S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16 && chunk == 64 && T > 0) {
        const size_t need = kda::prefill_split_workspace_bytes(N, T, H);
        if (!workspace || ws_bytes < need) return KDA_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_ALIGN;
        return cuda_status(kda::launch_prefill_split_ws(q, k, v, g, beta, S0, o, S_out, cu_seqlens,
                                                        N, T, H, workspace, s));
    }
    // the CUDA-core kernel needs no workspace
    return cuda_status(kda::launch_prefill_simt(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, T, H,
                                                chunk, dtype == KDA_BF16, s));
}

int kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                    const float *beta, float *S_inout, float *o, int B, int H, int dk, int dv,
                    int dtype, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || B < 0 || H < 1) return KDA_ERR_DIM;
    if ((int64_t)B * H * 2 >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S_inout || !o) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S_inout, o};
    for (const void *p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(kda::launch_decode(q, k, v, g, beta, S_inout, o, B, H, dtype == KDA_BF16, s));
}

int kda_decode_step_pool(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, void *S_pool, int state_dtype,
                         const int32_t *state_indices, int P, float *o, int B, int H, int dk,
                         int dv, int dtype, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (state_dtype != KDA_BF16 && state_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || B < 0 || H < 1 || P < 0) return KDA_ERR_DIM;
    if ((int64_t)B * H * 2 >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (!state_indices && P < B) return KDA_ERR_DIM;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S_pool || !o) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S_pool, o, state_indices};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(kda::launch_decode_pool(q, k, v, g, beta, S_pool, state_dtype == KDA_BF16,
                                               state_indices, P, o, B, H, dtype == KDA_BF16, s));
}

int kda_conv_prologue(const void *xq, const void *xk, const void *xv, const float *conv_w,
                      const void *conv_in, void *conv_out, void *q, void *k, void *v,
                      const int32_t *cu_seqlens, int N, int64_t T, int H, int d, float q_scale,
                      float eps, void *stream) {
    if (d != kda::kDK || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (!(eps >= 0.f) || !(q_scale == q_scale) || q_scale - q_scale != 0.f) return KDA_ERR_VALUE;
    if (!cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!xq || !xk || !xv || !conv_w || !q || !k || !v)) return KDA_ERR_NULL;
    if (conv_in && conv_in == conv_out) return KDA_ERR_VALUE;
    const void *ptrs[] = {xq, xk, xv, conv_w, conv_in, conv_out, q, k, v, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    if (T == 0 && !conv_out) return KDA_OK;
    return cuda_status(kda::launch_conv_prologue(xq, xk, xv, conv_w, conv_in, conv_out, q, k, v,
                                                 cu_seqlens, N, T, H, q_scale, eps,
                                                 static_cast<cudaStream_t>(stream)));
}

int kda_prefill_chunked_gated(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const float *S0, const void *gate,
                              const float *norm_w, float eps, float *out, float *S_out,
                              const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                              int chunk, int dtype, void *stream) {
    if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_CHUNK;
    if (!(eps >= 0.f)) return KDA_ERR_VALUE;
    if (!S_out || !cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!q || !k || !v || !g || !beta || !gate || !norm_w || !out)) return KDA_ERR_NULL;
    const void *ptrs[] = {q, k, v, g, beta, S0, gate, norm_w, out, S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16 && chunk == 64 && T > 0) {
        const cudaError_t e = kda::launch_prefill_split_gated(q, k, v, g, beta, S0, gate, norm_w, eps,
                                                              out, S_out, cu_seqlens, N, T, H, s);
        return e == cudaErrorMemoryAllocation ? KDA_ERR_WORKSPACE : cuda_status(e);
    }
    // CUDA-core prefill into `out`, then the gated norm in place
    cudaError_t e = kda::launch_prefill_simt(q, k, v, g, beta, S0, out, S_out, cu_seqlens, N, T, H,
                                             chunk, dtype == KDA_BF16, s);
    if (e == cudaSuccess) e = kda::launch_gated_norm(out, gate, norm_w, eps, T * H, s);
    return cuda_status(e);
}

int kda_layer_prefill(const void *xq, const void *xk, const void *xv, const float *conv_w,
                      const void *conv_in, void *conv_out, const float *g, const float *beta,
                      const float *S0, const void *gate, const float *norm_w, float q_scale,
                      float l2_eps, float norm_eps, float *out, float *S_out,
                      const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                      void *stream) {
    if (dk != kda::kDK || dv != kda::kDV || N < 1 || H < 1 || T < 0 || T >= (int64_t(1) << 31))
        return KDA_ERR_DIM;
    if ((int64_t)N * H * (kda::kDV / 32) >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (!(l2_eps >= 0.f) || !(norm_eps >= 0.f) || !(q_scale == q_scale) || q_scale - q_scale != 0.f)
        return KDA_ERR_VALUE;
    if (conv_in && conv_in == conv_out) return KDA_ERR_VALUE;
    if (!S_out || !cu_seqlens) return KDA_ERR_NULL;
    if (T > 0 && (!xq || !xk || !xv || !conv_w || !g || !beta || !gate || !norm_w || !out))
        return KDA_ERR_NULL;
    const void *ptrs[] = {xq, xk, xv, conv_w, conv_in, conv_out, g, beta, S0, gate, norm_w, out,
                          S_out, cu_seqlens};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {   // every sequence empty: windows and states pass through
        cudaError_t e = cudaSuccess;
        if (conv_out)
            e = kda::launch_conv_prologue(xq, xk, xv, conv_w, conv_in, conv_out, nullptr, nullptr,
                                          nullptr, cu_seqlens, N, T, H, q_scale, l2_eps, s);
        if (e == cudaSuccess)
            e = kda::launch_prefill_simt(nullptr, nullptr, nullptr, g, beta, S0, out, S_out,
                                         cu_seqlens, N, T, H, 64, true, s);
        return cuda_status(e);
    }
    const cudaError_t e = kda::launch_prefill_layer(xq, xk, xv, conv_w, conv_in, conv_out, g, beta,
                                                    S0, gate, norm_w, q_scale, l2_eps, norm_eps,
                                                    out, S_out, cu_seqlens, N, T, H, s);
    return e == cudaErrorMemoryAllocation ? KDA_ERR_WORKSPACE : cuda_status(e);
}

int kda_decode_layer_step(const void *xq, const void *xk, const void *xv, const float *conv_w,
                          void *conv_pool, const float *g, const float *beta, const void *gate,
                          const float *norm_w, void *S_pool, int state_dtype,
                          const int32_t *state_indices, int P, float *out, int B, int H, int dk,
                          int dv, float q_scale, float l2_eps, float norm_eps, void *stream) {
    if (state_dtype != KDA_BF16 && state_dtype != KDA_F32) return KDA_ERR_DTYPE;
    if (dk != kda::kDK || dv != kda::kDV || B < 0 || H < 1 || P < 0) return KDA_ERR_DIM;
    if ((int64_t)B * H >= (int64_t(1) << 31)) return KDA_ERR_DIM;
    if (!state_indices && P < B) return KDA_ERR_DIM;
    if (!(l2_eps >= 0.f) || !(norm_eps >= 0.f) || !(q_scale == q_scale) || q_scale - q_scale != 0.f)
        return KDA_ERR_VALUE;
    if (B == 0) return KDA_OK;
    if (!xq || !xk || !xv || !conv_w || !conv_pool || !g || !beta || !gate || !norm_w || !S_pool || !out)
        return KDA_ERR_NULL;
    const void *ptrs[] = {xq, xk, xv, conv_w, conv_pool, g, beta, gate, norm_w, S_pool, state_indices, out};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGN;
    return cuda_status(kda::launch_decode_layer(xq, xk, xv, conv_w, conv_pool, g, beta, gate, norm_w,
                                                S_pool, state_dtype == KDA_BF16, state_indices, P,
                                                out, B, H, q_scale, l2_eps, norm_eps,
                                                static_cast<cudaStream_t>(stream)));
}

int kda_workspace_release(void) { return cuda_status(kda::release_workspace_pool()); }

int kda_device_error(unsigned int *code, int reset) {
    if (!code) return KDA_ERR_NULL;
    unsigned int a = 0, b = 0, c = 0, d = 0;
    const cudaError_t e1 = kda::read_device_error(&a, reset != 0);
    const cudaError_t e2 = kda::read_decode_error(&b, reset != 0);
    const cudaError_t e3 = kda::read_layer_error(&c, reset != 0);
    const cudaError_t e4 = kda::read_simt_error(&d, reset != 0);
    *code = a | b | c | d;
    const cudaError_t e = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : (e3 != cudaSuccess ? e3 : e4));
    return cuda_status(e);
}

}  // extern "C"
