// Chunked KDA prefill on fp32 CUDA cores (FFMA): any chunk size in {16, 32,
// 64}, bf16 or fp32 q/k/v.  It is the path for fp32 inputs (where fp32
// accumulation throughout is needed) and for chunk sizes the tensor-core
// path does not take.
//
// The recurrence ("Colibri Kimi K3 Metal backend", architecture section)
//   S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,
//   o_t = S_t^T q_t
// unrolled over a chunk of L tokens with b_r = sum_{t<=r} g_t gives
//   G^kk_rs = sum_c k_rc k_sc e^{b_rc - b_sc} (s < r),  G^qk_rs likewise (s <= r)
//   (I + Diag(beta) G^kk) U = Diag(beta) (V - K0 S),   K0_r = e^{b_r} * k_r
//   O = Q0 S + G^qk U,                                 Q0_r = e^{b_r} * q_r
//   S <- Diag(e^{b_L}) S + Kbar^T U,                   Kbar_s = e^{b_L - b_s} * k_s
// Every pairwise factor e^{b_r - b_s} (s <= r) is evaluated directly, so no
// factor ever exceeds 1.
//
// Work split: one block per (sequence, head, value-slice of DVS columns);
// value columns of S evolve independently.  The block walks its sequence's
// chunks in order, keeping its fp32 state slice in shared memory.
#include "kda_internal.h"

namespace kda {

// Set (bit 0) when a block finds its sequence's cu_seqlens entries outside
// [0, T] or decreasing: its tokens are then clamped to [0, T).
__device__ unsigned int g_kda_simt_error = 0;

namespace {

constexpr int kSimtThreads = 256;

template <int C, int DVS>
struct SimtSmem {
    static constexpr int LD = kDK + 1;   // padded row stride of [C][DK] tiles
    static constexpr int LU = DVS + 4;   // row stride of [C][DVS] tiles
    static constexpr size_t floats =
        4 * (size_t)C * LD + 2 * (size_t)C * C + (size_t)kDK * DVS + (size_t)C * LU + C + kDK;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <typename TIn, int C, int DVS>
__global__ void __launch_bounds__(kSimtThreads, 1)
prefill_simt_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k,
                    const TIn *__restrict__ v, const float *__restrict__ g,
                    const float *__restrict__ beta, const float *__restrict__ S0,
                    float *__restrict__ o, float *S_out, const int32_t *__restrict__ cu,
                    int N, int H, int T) {
    using L = SimtSmem<C, DVS>;
    constexpr int LD = L::LD, LU = L::LU;
    constexpr int NSL = kDV / DVS;
    constexpr int NT = kSimtThreads;
    static_assert(DVS == 32, "thread mappings below assume 32-column slices");

    extern __shared__ float smem[];
    float *sK = smem;                 // [C][LD]  k, then Kbar
    float *sQ = sK + C * LD;          // [C][LD]  q, then Q0
    float *sB = sQ + C * LD;          // [C][LD]  cumulative log-decay b
    float *sK0 = sB + C * LD;         // [C][LD]  e^{b} k
    float *sM = sK0 + C * LD;         // [C][C]   beta_r G^kk_rs (s < r)
    float *sA = sM + C * C;           // [C][C]   G^qk_rs (s <= r)
    float *sS = sA + C * C;           // [DK][DVS] state slice
    float *sU = sS + kDK * DVS;       // [C][LU]  V, then R = V - K0 S, then U
    float *sBeta = sU + C * LU;       // [C]
    float *sGam = sBeta + C;          // [DK] e^{b_L}
    __shared__ int s_seq;

    const int t = threadIdx.x;
    const int slice = blockIdx.x % NSL;
    const int h = (blockIdx.x / NSL) % H;
    const int rank = blockIdx.x / (NSL * H);
    const int n = lpt_sequence(cu, N, rank, &s_seq);
    // tokens clamped to [0, T): an inconsistent cu_seqlens (cu[N] != T, a
    // caller error) never makes the kernel read or write past the buffers
    const int tok0 = min(max(cu[n], 0), T);
    const int len = min(max(cu[n + 1], tok0), T) - tok0;
    if (t == 0 && (cu[n] != tok0 || cu[n + 1] != tok0 + len)) atomicOr(&g_kda_simt_error, kErrWait);
    const int col0 = slice * DVS;
    const size_t st_off = ((size_t)n * H + h) * kDK * kDV + col0;

    for (int idx = t; idx < kDK * DVS; idx += NT) {
        const int i = idx / DVS, j = idx % DVS;
        sS[idx] = S0 ? S0[st_off + (size_t)i * kDV + j] : 0.f;
    }

    const int lane = t & 31, warp = t >> 5;

    for (int c0 = 0; c0 < len; c0 += C) {
        const int Lc = min(C, len - c0);
        // ---- load the chunk ------------------------------------------------
        for (int idx = t; idx < C * kDK; idx += NT) {
            const int r = idx / kDK, c = idx % kDK;
            float kv = 0.f, qv = 0.f;
            if (r < Lc) {
                const size_t gi = ((size_t)(tok0 + c0 + r) * H + h) * kDK + c;
                kv = load_in(k, gi);
                qv = load_in(q, gi);
            }
            sK[r * LD + c] = kv;
            sQ[r * LD + c] = qv;
        }
        for (int idx = t; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            sU[r * LU + j] = (r < Lc) ? load_in(v, ((size_t)(tok0 + c0 + r) * H + h) * kDV + col0 + j)
                                      : 0.f;
        }
        if (t < C) sBeta[t] = (t < Lc) ? beta[(size_t)(tok0 + c0 + t) * H + h] : 0.f;
        if (t < kDK) {
            float acc = 0.f;
            for (int r = 0; r < C; ++r) {
                if (r < Lc) acc += g[((size_t)(tok0 + c0 + r) * H + h) * kDK + t];
                sB[r * LD + t] = acc;
            }
            sGam[t] = expf(acc);
        }
        __syncthreads();

        // ---- gated Gram matrices ------------------------------------------
        for (int p = t; p < C * C; p += NT) {
            const int r = p / C, s = p % C;
            float gk = 0.f, gq = 0.f;
            if (r < Lc && s <= r) {
                const float *kr = sK + r * LD, *ks = sK + s * LD, *qr = sQ + r * LD;
                const float *br = sB + r * LD, *bs = sB + s * LD;
#pragma unroll 4
                for (int c = 0; c < kDK; ++c) {
                    const float kse = ks[c] * expf(br[c] - bs[c]);
                    gk += kr[c] * kse;
                    gq += qr[c] * kse;
                }
            }
            sM[p] = (s < r) ? sBeta[r] * gk : 0.f;
            sA[p] = gq;
        }
        __syncthreads();

        // ---- decay-folded operands ----------------------------------------
        for (int idx = t; idx < C * kDK; idx += NT) {
            const int r = idx / kDK, c = idx % kDK;
            const float b = sB[r * LD + c];
            const float bL = sB[(Lc - 1) * LD + c];
            const float eb = expf(b);
            const float kv = sK[r * LD + c];
            sK0[r * LD + c] = kv * eb;
            sQ[r * LD + c] *= eb;
            sK[r * LD + c] = kv * expf(bL - b);     // rows >= Lc are zero
        }
        __syncthreads();

        // ---- R = V - K0 S  (rows r = warp + 8m, column = lane) --------------
        {
            float acc[C / 8];
#pragma unroll
            for (int m = 0; m < C / 8; ++m) acc[m] = 0.f;
            for (int c = 0; c < kDK; ++c) {
                const float sv = sS[c * DVS + lane];
#pragma unroll
                for (int m = 0; m < C / 8; ++m) acc[m] += sK0[(warp + 8 * m) * LD + c] * sv;
            }
#pragma unroll
            for (int m = 0; m < C / 8; ++m) sU[(warp + 8 * m) * LU + lane] -= acc[m];
        }
        __syncthreads();

        // ---- forward substitution (I + M) U = Diag(beta) R -----------------
        // 8 lanes per column: lane group (warp, lane % 4) owns column
        // 4 * warp + lane % 4; part = lane / 4 sums rows s = part (mod 8).
        {
            const int col = 4 * warp + (lane & 3);
            const int part = lane >> 2;
            for (int r = 0; r < Lc; ++r) {
                float acc = 0.f;
                for (int s = part; s < r; s += 8) acc += sM[r * C + s] * sU[s * LU + col];
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                acc += __shfl_xor_sync(0xffffffffu, acc, 8);
                acc += __shfl_xor_sync(0xffffffffu, acc, 16);
                const float u = sBeta[r] * sU[r * LU + col] - acc;
                __syncwarp();
                if (part == 0) sU[r * LU + col] = u;
                __syncwarp();
            }
        }
        __syncthreads();

        // ---- O = Q0 S + G^qk U  ->  o ---------------------------------------
        {
            float acc[C / 8];
#pragma unroll
            for (int m = 0; m < C / 8; ++m) acc[m] = 0.f;
            for (int c = 0; c < kDK; ++c) {
                const float sv = sS[c * DVS + lane];
#pragma unroll
                for (int m = 0; m < C / 8; ++m) acc[m] += sQ[(warp + 8 * m) * LD + c] * sv;
            }
            for (int s = 0; s < Lc; ++s) {
                const float uv = sU[s * LU + lane];
#pragma unroll
                for (int m = 0; m < C / 8; ++m) acc[m] += sA[(warp + 8 * m) * C + s] * uv;
            }
#pragma unroll
            for (int m = 0; m < C / 8; ++m) {
                const int r = warp + 8 * m;
                if (r < Lc)
                    o[((size_t)KDA_DBG_INDEX(g_kda_simt_error, tok0 + c0 + r, 0, T) * H + h) * kDV + col0 +
                      lane] = acc[m];
            }
        }
        __syncthreads();

        // ---- S <- Diag(e^{b_L}) S + Kbar^T U  (rows c = warp + 8m) ---------
        {
            float acc[kDK / 8];
#pragma unroll
            for (int m = 0; m < kDK / 8; ++m) acc[m] = sGam[warp + 8 * m] * sS[(warp + 8 * m) * DVS + lane];
            for (int r = 0; r < Lc; ++r) {
                const float uv = sU[r * LU + lane];
#pragma unroll
                for (int m = 0; m < kDK / 8; ++m) acc[m] += sK[r * LD + warp + 8 * m] * uv;
            }
#pragma unroll
            for (int m = 0; m < kDK / 8; ++m) sS[(warp + 8 * m) * DVS + lane] = acc[m];
        }
        __syncthreads();
    }

    for (int idx = t; idx < kDK * DVS; idx += NT) {
        const int i = idx / DVS, j = idx % DVS;
        S_out[st_off + (size_t)i * kDV + j] = sS[idx];
    }
}

template <typename TIn, int C>
cudaError_t launch_c(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, const float *S0, float *o, float *S_out,
                     const int32_t *cu, int N, int H, int T, cudaStream_t stream) {
    constexpr int DVS = 32;
    using L = SimtSmem<C, DVS>;
    auto kern = prefill_simt_kernel<TIn, C, DVS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)N * H * (kDV / DVS);
    kern<<<(unsigned)blocks, kSimtThreads, L::bytes, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v), g,
        beta, S0, o, S_out, cu, N, H, T);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_t(int chunk, const void *q, const void *k, const void *v, const float *g,
                     const float *beta, const float *S0, float *o, float *S_out,
                     const int32_t *cu, int N, int H, int T, cudaStream_t stream) {
    switch (chunk) {
        case 16: return launch_c<TIn, 16>(q, k, v, g, beta, S0, o, S_out, cu, N, H, T, stream);
        case 32: return launch_c<TIn, 32>(q, k, v, g, beta, S0, o, S_out, cu, N, H, T, stream);
        default: return launch_c<TIn, 64>(q, k, v, g, beta, S0, o, S_out, cu, N, H, T, stream);
    }
}

}  // namespace

cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, const float *S0, float *o, float *S_out,
                                const int32_t *cu_seqlens, int N, int64_t T, int H, int chunk,
                                bool bf16, cudaStream_t stream) {
    if (bf16)
        return launch_t<__nv_bfloat16>(chunk, q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, H,
                                       (int)T, stream);
    return launch_t<float>(chunk, q, k, v, g, beta, S0, o, S_out, cu_seqlens, N, H, (int)T, stream);
}

cudaError_t read_simt_error(unsigned int *code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_kda_simt_error, sizeof(unsigned int));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_kda_simt_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
