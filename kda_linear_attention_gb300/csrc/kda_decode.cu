// Fused KDA decode step: one token per sequence, state updated in place.
//
// Per (b, h) the token step of "Colibri Kimi K3 Metal backend", section 8.2,
// done in one pass over the state:
//   a_i = exp(g_i);  S'_ij = a_i S_ij                        (row decay)
//   u_j = sum_i k_i S'_ij;  w_j = beta (v_j - u_j)           (prediction, delta)
//   S_ij <- S'_ij + k_i w_j                                  (rank-1 update)
//   o_j = sum_i q_i S_ij = sum_i q_i S'_ij + (q.k) w_j       (readout, updated S)
// The last identity lets both column reductions run on the decayed state
// while it is still in registers, so each 64 KiB state is read once and
// written once: the kernel is bound by HBM bandwidth.
//
// The state can live in a pool addressed by per-sequence slots (continuous
// batching: sequence b uses pool row state_indices[b], a negative slot marks
// a padding row that is skipped), and can be stored in bf16 (loaded into
// fp32, updated in fp32, rounded to nearest-even on the store).
//
// Work split: a block owns COLS value-columns of one (b, h) state (columns
// evolve independently).  Thread t holds float4 column group t % (COLS/4) for
// rows rg, rg + NRG, ... (rg = t / (COLS/4)), so each warp load covers whole
// 128-bit-coalesced row segments.  Column sums are reduced across row groups
// through shared memory, each (component, column) sum taken by one thread.
#include "kda_internal.h"

namespace kda {

// Set (bit 1) when a decode slot index lies past the end of the pool.
__device__ unsigned int g_kda_decode_error = 0;

namespace {

constexpr int kDecodeThreads = 256;

// four consecutive fp32 state values <-> registers (streaming)
__device__ __forceinline__ float4 load_state4(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void store_state4(float *p, float4 x) {
    __stcs(reinterpret_cast<float4 *>(p), x);
}

template <typename TIn, typename TS, int COLS>
__global__ void __launch_bounds__(kDecodeThreads, (COLS == 128 ? 2 : 4))
decode_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
              const float *__restrict__ g, const float *__restrict__ beta,
              TS *__restrict__ S, float *__restrict__ o, const int32_t *__restrict__ slots,
              int H, int P) {
    constexpr int C4 = COLS / 4;                 // float4 column groups per block
    constexpr int NRG = kDecodeThreads / C4;     // row groups
    constexpr int RPT = kDK / NRG;               // rows per thread
    constexpr int NSPLIT = kDV / COLS;           // blocks per state

    const int unit = blockIdx.x / NSPLIT;        // b * H + h
    const int cs = blockIdx.x % NSPLIT;
    const int t = threadIdx.x;
    const int c4 = t % C4;
    const int rg = t / C4;
    const int col0 = cs * COLS + c4 * 4;

    // pool row of this sequence (the identity without a slot table)
    int slot = unit / H;
    if (slots) {
        slot = slots[unit / H];
        if (slot < 0 || slot >= P) {             // padding row (or an invalid slot)
            if (slot >= P && t == 0) atomicOr(&g_kda_decode_error, 2u);
            if (rg == 0)
                *reinterpret_cast<float4 *>(o + (size_t)unit * kDV + col0) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            return;
        }
    }
    slot = KDA_DBG_INDEX(g_kda_decode_error, slot, 0, P);
    TS *Su = S + ((size_t)slot * H + unit % H) * kDK * kDV;

    // Issue the state loads first; they are independent of everything else.
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = load_state4(Su + (size_t)(rg + r * NRG) * kDV + col0);

    __shared__ float sq[kDK], sk[kDK], sa[kDK];
    __shared__ float red[8][NRG][C4];            // row-group partials: k^T S (x..w), q^T S (x..w)
    __shared__ float tot[8][C4];                 // their sums over the row groups
    __shared__ float s_qk[kDK / 32];

    if (t < kDK) {
        const float qi = load_in(q, (size_t)unit * kDK + t);
        const float ki = load_in(k, (size_t)unit * kDK + t);
        sq[t] = qi;
        sk[t] = ki;
        sa[t] = expf(g[(size_t)unit * kDK + t]);
        float p = qi * ki;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if ((t & 31) == 0) s_qk[t >> 5] = p;
    }
    __syncthreads();

    float4 uk = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 uq = uk;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int i = rg + r * NRG;
        const float a = sa[i], ki = sk[i], qi = sq[i];
        s[r].x *= a; s[r].y *= a; s[r].z *= a; s[r].w *= a;
        uk.x += ki * s[r].x; uk.y += ki * s[r].y; uk.z += ki * s[r].z; uk.w += ki * s[r].w;
        uq.x += qi * s[r].x; uq.y += qi * s[r].y; uq.z += qi * s[r].z; uq.w += qi * s[r].w;
    }
    // the column sums over the row groups: each of 8 * C4 threads sums one
    // (component, column group) once, then every thread reads its 8 totals
    red[0][rg][c4] = uk.x; red[1][rg][c4] = uk.y; red[2][rg][c4] = uk.z; red[3][rg][c4] = uk.w;
    red[4][rg][c4] = uq.x; red[5][rg][c4] = uq.y; red[6][rg][c4] = uq.z; red[7][rg][c4] = uq.w;
    __syncthreads();
    if (t < 8 * C4) {
        const int comp = t / C4, cc = t % C4;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < NRG; ++j) sum += red[comp][j][cc];
        tot[comp][cc] = sum;
    }
    __syncthreads();
    const float4 Uk = make_float4(tot[0][c4], tot[1][c4], tot[2][c4], tot[3][c4]);
    const float4 Uq = make_float4(tot[4][c4], tot[5][c4], tot[6][c4], tot[7][c4]);
    float qk = 0.f;
#pragma unroll
    for (int j = 0; j < kDK / 32; ++j) qk += s_qk[j];

    const float bt = beta[unit];
    const size_t vo = (size_t)unit * kDV + col0;
    float4 w;
    w.x = bt * (load_in(v, vo + 0) - Uk.x);
    w.y = bt * (load_in(v, vo + 1) - Uk.y);
    w.z = bt * (load_in(v, vo + 2) - Uk.z);
    w.w = bt * (load_in(v, vo + 3) - Uk.w);

#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int i = rg + r * NRG;
        const float ki = sk[i];
        s[r].x += ki * w.x; s[r].y += ki * w.y; s[r].z += ki * w.z; s[r].w += ki * w.w;
        store_state4(Su + (size_t)i * kDV + col0, s[r]);
    }
    if (rg == 0) {
        float4 ov;
        ov.x = Uq.x + qk * w.x; ov.y = Uq.y + qk * w.y;
        ov.z = Uq.z + qk * w.z; ov.w = Uq.w + qk * w.w;
        *reinterpret_cast<float4 *>(o + vo) = ov;
    }
}

// ----------------------------------------------------------------------------
// bf16-stored states: the state is kept packed (two bf16 per register) from
// the load to the store and unpacked where it is used, so a thread keeps 128
// bytes of state in flight with 32 registers.  One block per (b, h); thread
// t holds columns 8 (t % 16) .. + 7 of rows t / 16 + 16 r, r < 8 (a 16-byte
// load per row).  The decay is applied twice (once for the column sums, once
// for the update), both times from the stored values.
// ----------------------------------------------------------------------------
constexpr int kPackedThreads = 256;

__device__ __forceinline__ void unpack8_bf16(uint4 u, float (&x)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
__device__ __forceinline__ uint4 pack8_bf16(const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename TIn>
__global__ void __launch_bounds__(kPackedThreads, 3)
decode_bf16_state_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                         const float *__restrict__ g, const float *__restrict__ beta,
                         __nv_bfloat16 *__restrict__ S, float *__restrict__ o,
                         const int32_t *__restrict__ slots, int H, int P) {
    constexpr int C8 = 16;                       // 8-column groups
    constexpr int NRG = kPackedThreads / C8;     // 16 row groups
    constexpr int RPT = kDK / NRG;               // 8 rows per thread
    const int unit = blockIdx.x;                 // b * H + h
    const int t = threadIdx.x;
    const int c8 = t % C8, rg = t / C8;
    const int col0 = 8 * c8;

    int slot = unit / H;
    if (slots) {
        slot = slots[unit / H];
        if (slot < 0 || slot >= P) {             // padding row (or an invalid slot)
            if (slot >= P && t == 0) atomicOr(&g_kda_decode_error, 2u);
            if (rg == 0) {
                float4 *op = reinterpret_cast<float4 *>(o + (size_t)unit * kDV + col0);
                op[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                op[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            return;
        }
    }
    slot = KDA_DBG_INDEX(g_kda_decode_error, slot, 0, P);
    __nv_bfloat16 *Su = S + ((size_t)slot * H + unit % H) * kDK * kDV;
    uint4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        s[r] = __ldcs(reinterpret_cast<const uint4 *>(Su + (size_t)(rg + r * NRG) * kDV + col0));

    __shared__ float sq[kDK], sk[kDK], sa[kDK];
    __shared__ float red[16][NRG][C8];           // partials: k^T S (8 columns), q^T S (8 columns)
    __shared__ float tot[16][C8];
    __shared__ float s_qk[kDK / 32];
    if (t < kDK) {
        const float qi = load_in(q, (size_t)unit * kDK + t);
        const float ki = load_in(k, (size_t)unit * kDK + t);
        sq[t] = qi;
        sk[t] = ki;
        sa[t] = expf(g[(size_t)unit * kDK + t]);
        float pq = qi * ki;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) pq += __shfl_xor_sync(0xffffffffu, pq, off);
        if ((t & 31) == 0) s_qk[t >> 5] = pq;
    }
    __syncthreads();

    float uk[8], uq[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) uk[c] = uq[c] = 0.f;
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int i = rg + r * NRG;
        const float a = sa[i], ki = sk[i], qi = sq[i];
        float x[8];
        unpack8_bf16(s[r], x);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float xd = x[c] * a;
            uk[c] = fmaf(ki, xd, uk[c]);
            uq[c] = fmaf(qi, xd, uq[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        red[c][rg][c8] = uk[c];
        red[8 + c][rg][c8] = uq[c];
    }
    __syncthreads();
    {
        // 256 threads: one (component, column group) sum each
        const int comp = t / C8, cc = t % C8;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < NRG; ++j) sum += red[comp][j][cc];
        tot[comp][cc] = sum;
    }
    __syncthreads();
    float qk = 0.f;
#pragma unroll
    for (int j = 0; j < kDK / 32; ++j) qk += s_qk[j];
    const float bt = beta[unit];
    const size_t vo = (size_t)unit * kDV + col0;
    float w[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) w[c] = bt * (load_in(v, vo + c) - tot[c][c8]);

#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int i = rg + r * NRG;
        const float a = sa[i], ki = sk[i];
        float x[8];
        unpack8_bf16(s[r], x);
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = fmaf(ki, w[c], x[c] * a);
        __stcs(reinterpret_cast<uint4 *>(Su + (size_t)i * kDV + col0), pack8_bf16(x));
    }
    if (rg == 0) {
        float ov[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) ov[c] = tot[8 + c][c8] + qk * w[c];
        float4 *op = reinterpret_cast<float4 *>(o + vo);
        op[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
        op[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
    }
}

template <typename TIn, typename TS>
cudaError_t launch_typed(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, void *S, float *o, const int32_t *slots, int B, int H,
                         int P, cudaStream_t stream) {
    // Two blocks per state (64 columns each): twice the blocks of a
    // whole-state split, a shorter tail and fewer registers per thread.
    constexpr int COLS = 64;
    const long long units = (long long)B * H;
    const long long blocks = units * (kDV / COLS);
    decode_kernel<TIn, TS, COLS><<<(unsigned)blocks, kDecodeThreads, 0, stream>>>(
        static_cast<const TIn *>(q), static_cast<const TIn *>(k), static_cast<const TIn *>(v),
        g, beta, static_cast<TS *>(S), o, slots, H, P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *S, float *o, int B, int H, bool bf16,
                          cudaStream_t stream) {
    if (bf16) return launch_typed<__nv_bfloat16, float>(q, k, v, g, beta, S, o, nullptr, B, H, B, stream);
    return launch_typed<float, float>(q, k, v, g, beta, S, o, nullptr, B, H, B, stream);
}

cudaError_t launch_decode_pool(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, void *S_pool, bool state_bf16,
                               const int32_t *slots, int P, float *o, int B, int H, bool bf16,
                               cudaStream_t stream) {
    if (state_bf16) {
        // the packed kernel: one block per state
        const long long units = (long long)B * H;
        if (bf16)
            decode_bf16_state_kernel<__nv_bfloat16><<<(unsigned)units, kPackedThreads, 0, stream>>>(
                static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                static_cast<const __nv_bfloat16 *>(v), g, beta, static_cast<__nv_bfloat16 *>(S_pool), o,
                slots, H, P);
        else
            decode_bf16_state_kernel<float><<<(unsigned)units, kPackedThreads, 0, stream>>>(
                static_cast<const float *>(q), static_cast<const float *>(k), static_cast<const float *>(v),
                g, beta, static_cast<__nv_bfloat16 *>(S_pool), o, slots, H, P);
        return cudaGetLastError();
    }
    if (bf16) {
        return launch_typed<__nv_bfloat16, float>(q, k, v, g, beta, S_pool, o, slots, B, H, P, stream);
    }
    return launch_typed<float, float>(q, k, v, g, beta, S_pool, o, slots, B, H, P, stream);
}

cudaError_t read_decode_error(unsigned int *code, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_kda_decode_error, sizeof(unsigned int));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_kda_decode_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
