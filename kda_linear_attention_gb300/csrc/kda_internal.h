// Internal launcher interface of libkda_gb300 (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr int kDK = 128;
constexpr int kDV = 128;

// Bits of the device error word (kda_device_error).
constexpr unsigned kErrWait = 1u;        // a bounded wait gave up, or cu_seqlens broke the call's precondition
constexpr unsigned kErrSlot = 2u;        // a pool slot index past the end of the pool
constexpr unsigned kErrGateRange = 4u;   // the tensor-core prefill saw a gate g outside [-5, 0] (or NaN)
constexpr unsigned kErrBounds = 8u;      // debug builds (KDA_DEBUG): an index check failed; the access was kept in bounds
constexpr unsigned kErrFp16Range = 16u;  // the tensor-core prefill's u left fp16's finite range (|u| >= 65504 or NaN)
// Lower bound of the log-decay gate that the decay folding of the
// tensor-core prefill is sized for (the model's gate lower bound).
constexpr float kGateMin = -5.0f;

// Debug builds (nvcc -DKDA_DEBUG; python -m kda_linear_attention_gb300.build
// --debug): index checks on the kernels' global-memory addressing, in place
// of a memory checker.  A failed check sets kErrBounds in the kernel's error
// word and replaces the index by the first value of its range, so the access
// stays inside the buffer (the outputs are then invalid, and flagged);
// nothing traps and no control flow changes.  Release builds compile the
// checks out.
#ifdef KDA_DEBUG
__device__ __forceinline__ long long dbg_index(unsigned int *word, long long i, long long lo,
                                               long long hi) {
    if (i < lo || i >= hi) {
        atomicOr(word, kErrBounds);
        return lo;
    }
    return i;
}
#define KDA_DBG_INDEX(word, i, lo, hi) \
    ((decltype(i))::kda::dbg_index(&(word), (long long)(i), (long long)(lo), (long long)(hi)))
#else
#define KDA_DBG_INDEX(word, i, lo, hi) (i)
#endif

// Fused decode step (kda_decode.cu).  Returns the launch error.
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *S, float *o, int B, int H, bool bf16,
                          cudaStream_t stream);

// Decode step on a state pool: sequence b updates pool row slots[b] (the
// identity when slots == nullptr; negative slots are padding rows whose o is
// zero); the pool is fp32 or bf16 (state_bf16).  P = pool rows.
cudaError_t launch_decode_pool(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, void *S_pool, bool state_bf16,
                               const int32_t *slots, int P, float *o, int B, int H, bool bf16,
                               cudaStream_t stream);
cudaError_t read_decode_error(unsigned int *code, bool reset);

// fp32 CUDA-core chunked prefill (kda_prefill_simt.cu): any chunk in {16,32,64},
// bf16 or fp32 inputs.
cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, const float *S0, float *o, float *S_out,
                                const int32_t *cu_seqlens, int N, int64_t T, int H, int chunk, bool bf16,
                                cudaStream_t stream);
// Error word of the CUDA-core prefill (bit 0: cu_seqlens outside [0, T] or
// decreasing; its tokens were clamped to [0, T)).
cudaError_t read_simt_error(unsigned int *code, bool reset);

// Two-kernel tensor-core chunked prefill (kda_prefill_split.cu): bf16 q/k/v,
// chunk 64, T >= 1.  Takes its workspace (see prefill_split_workspace_bytes)
// from a library-owned stream-ordered pool; returns cudaErrorMemoryAllocation
// when it cannot.
// `events` (optional, four timing events) are recorded on `stream` before
// the chunk plan, before the intra-chunk kernel, before the state pass and
// after it.
cudaError_t launch_prefill_split(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *S0, float *o, float *S_out,
                                 const int32_t *cu_seqlens, int N, int64_t T, int H,
                                 cudaStream_t stream, cudaEvent_t const *events = nullptr);
size_t prefill_split_workspace_bytes(int N, int64_t T, int H);

// The same prefill with its workspace in a fixed file-scope device array of
// kNoAllocScratchBytes (no allocation during the call); cudaErrorInvalidValue
// when the workspace the sizes need is larger.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
cudaError_t launch_prefill_split_noalloc(const void *q, const void *k, const void *v,
                                         const float *g, const float *beta, const float *S0,
                                         float *o, float *S_out, const int32_t *cu_seqlens, int N,
                                         int64_t T, int H, cudaStream_t stream);

// The same prefill with a workspace the caller owns (at least
// prefill_split_workspace_bytes(N, T, H) bytes, 256-byte aligned); nothing is
// allocated and nothing in it has to be cleared between calls.
cudaError_t launch_prefill_split_ws(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *S0, float *o, float *S_out,
                                    const int32_t *cu_seqlens, int N, int64_t T, int H, void *ws,
                                    cudaStream_t stream);

// Read (and optionally clear) the device-side error word that the
// tensor-core kernels set when a bounded wait gives up.
cudaError_t read_device_error(unsigned int *code, bool reset);
// Gives the current device's workspace pool memory back to the driver.
cudaError_t release_workspace_pool();

// The tensor-core prefill with the layer's gated RMSNorm fused into the state
// pass's output: out = RMSNorm(o) * norm_w * sigmoid(gate) instead of o
// (gate [T, H, 128] bf16, norm_w [128] fp32).
cudaError_t launch_prefill_split_gated(const void *q, const void *k, const void *v,
                                       const float *g, const float *beta, const float *S0,
                                       const void *gate, const float *norm_w, float eps,
                                       float *out, float *S_out, const int32_t *cu_seqlens, int N,
                                       int64_t T, int H, cudaStream_t stream,
                                       cudaEvent_t const *events = nullptr);

// The layer prefill on the tensor-core path: the conv prologue's q, k, v in
// a pool workspace (bf16), then the gated prefill on them (kda_layer.cu's
// prologue kernel, then this file's three launches).
cudaError_t launch_prefill_layer(const void *xq, const void *xk, const void *xv, const float *conv_w,
                                 const void *conv_in, void *conv_out, const float *g,
                                 const float *beta, const float *S0, const void *gate,
                                 const float *norm_w, float q_scale, float l2_eps, float norm_eps,
                                 float *out, float *S_out, const int32_t *cu_seqlens, int N,
                                 int64_t T, int H, cudaStream_t stream);

// The layer around the recurrence (kda_layer.cu).
// conv1d + SiLU on xq/xk/xv, L2 norm of q (times q_scale) and k; windows in
// and out [N, 3, 3, H, 128] bf16 (conv_in may be null: zeros; conv_out may
// be null: not written).
cudaError_t launch_conv_prologue(const void *xq, const void *xk, const void *xv, const float *conv_w,
                                 const void *conv_in, void *conv_out, void *q, void *k, void *v,
                                 const int32_t *cu_seqlens, int N, int64_t T, int H, float q_scale,
                                 float eps, cudaStream_t stream);
// In place over `rows` rows of 128: o <- RMSNorm(o) * norm_w * sigmoid(gate).
cudaError_t launch_gated_norm(float *o, const void *gate, const float *norm_w, float eps,
                              long long rows, cudaStream_t stream);
// Whole-layer decode step on slot-indexed pools (state fp32 or bf16, windows bf16).
cudaError_t launch_decode_layer(const void *xq, const void *xk, const void *xv, const float *conv_w,
                                void *conv_pool, const float *g, const float *beta, const void *gate,
                                const float *norm_w, void *S_pool, bool state_bf16,
                                const int32_t *slots, int P, float *out, int B, int H,
                                float q_scale, float l2_eps, float norm_eps, cudaStream_t stream);
cudaError_t read_layer_error(unsigned int *code, bool reset);

// The conv prologue's arithmetic, shared by the prologue kernel and the
// layer prefill that fuses it: bf16 pairs (low half = even channel) to and
// from float2 (exact / round to nearest even), and the SiLU of a channel
// pair, y / (1 + e^-y), with e^-y as a power of two and the hardware
// reciprocal (a few ulp; its results are rounded to bf16).
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float2 v) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float rcp_approx(float x) {   // 1 / x, about 1 ulp; 1 / inf = 0
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// 2^x on the special-function unit (ex2.approx, a few ulp; results below
// 2^-126 flush to 0, 2^x for x >= 128 is inf)
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// e^-y = 2^(-y log2 e), the pair's scaling in one packed multiply
__device__ __forceinline__ float2 silu2(float2 y) {
    const float2 a = __fmul2_rn(y, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    const float2 d = __fadd2_rn(make_float2(1.f, 1.f), make_float2(ex2_approx(a.x), ex2_approx(a.y)));
    return __fmul2_rn(y, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Input loads: bf16 or fp32 element -> fp32.
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }

// Longest-first placement of sequences onto blocks: the block whose sequence
// rank is `rank` processes the sequence with the rank-th largest length (ties
// by index), so the hardware block scheduler starts the longest sequences
// first.  For N above `kLptMaxN` the identity order is used.  Must be called
// by all threads of the block; `s_out` is a __shared__ int.
constexpr int kLptMaxN = 256;
__device__ __forceinline__ int lpt_sequence(const int32_t *cu, int N, int rank, int *s_out) {
    if (N > kLptMaxN) return rank;
    if (threadIdx.x == 0) *s_out = rank;   // fallback, overwritten below
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < N; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li) || (lj == li && j < i);
        }
        if (r == rank) *s_out = i;
    }
    __syncthreads();
    const int n = *s_out;
    __syncthreads();
    return n;
}

}  // namespace kda
