// C-ABI shim of libkda_gb300: argument validation and kernel dispatch.
// Declarations and the contract of each call are in include/kda.h.
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr int kVersion = 100;   // 0.1.0

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
        case KDA_ERR_WORKSPACE: return "workspace error";
        case KDA_ERR_CUDA: return "CUDA launch error";
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
    return cuda_status(kda::launch_prefill_simt(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, H,
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
    return cuda_status(kda::launch_prefill_simt(q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, H,
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

int kda_device_error(unsigned int *code, int reset) {
    if (!code) return KDA_ERR_NULL;
    unsigned int a = 0, b = 0;
    const cudaError_t e1 = kda::read_device_error(&a, reset != 0);
    const cudaError_t e2 = kda::read_decode_error(&b, reset != 0);
    *code = a | b;
    return cuda_status(e1 != cudaSuccess ? e1 : e2);
}

}  // extern "C"
