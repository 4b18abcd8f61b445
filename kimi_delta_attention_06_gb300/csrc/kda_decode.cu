// kda_decode.cu -- single-token KDA decode step, one CTA per (sequence, head).
//
// Per head the step is (KDA recurrence, SemiAnalysis Kimi K3 primer, wiki
// summary, section 1; cost model in section 2: ~7 D^2 FLOPs against 8 D^2
// bytes of fp32 state):
//
//   S'  = Diag(alpha) S                    alpha = exp(log_alpha)
//   u   = v - S'^T k
//   S   = S' + beta k u^T                  (written back in place)
//   o   = S^T q = S'^T q + beta (q . k) u
//
// The state is the only large operand, so the kernel is a single streaming
// pass: every thread issues its 128-bit loads of S up front, the two column
// reductions (S'^T k and S'^T q) run on registers + shared memory, and the
// same registers are written back.  No other global traffic of note.
#include "common.cuh"

namespace kda {

template <int D, int WARPS>
struct DecodeShape {
    static constexpr int kThreads = WARPS * 32;
    static constexpr int kLanesPerRow = D / 4;            // float4 per row
    static constexpr int kRowsPerIter = 32 / kLanesPerRow; // rows a warp covers per load
    static constexpr int kRowsPerWarp = D / WARPS;
    static constexpr int kIters = kRowsPerWarp / kRowsPerIter;
    static_assert(kRowsPerWarp % kRowsPerIter == 0, "shape");
};

// The two per-row updates of the step, on two-lane fp32 instructions (each lane rounds as
// the scalar fma / mul; the single-token and K-token kernels share them, so a one-token
// commit reproduces the single-token step bit for bit):
//   r1 += (alpha k)_row * S[row, 4 columns],  r2 += (alpha q)_row * S[row, 4 columns]
__device__ __forceinline__ void col_sums(float4& r1, float4& r2, float ak, float aq, float4 x) {
    const float2 ak2 = make_float2(ak, ak), aq2 = make_float2(aq, aq);
    const float2 xl = make_float2(x.x, x.y), xh = make_float2(x.z, x.w);
    const float2 r1l = ffma2(ak2, xl, make_float2(r1.x, r1.y)), r1h = ffma2(ak2, xh, make_float2(r1.z, r1.w));
    const float2 r2l = ffma2(aq2, xl, make_float2(r2.x, r2.y)), r2h = ffma2(aq2, xh, make_float2(r2.z, r2.w));
    r1 = make_float4(r1l.x, r1l.y, r1h.x, r1h.y);
    r2 = make_float4(r2l.x, r2l.y, r2h.x, r2h.y);
}
//   S[row, 4 columns] = alpha_row S[row, 4 columns] + (beta k_row) u[4 columns]
__device__ __forceinline__ float4 state_update(float4 x, float a, float kr, float4 u) {
    const float2 a2 = make_float2(a, a), k2 = make_float2(kr, kr);
    const float2 lo = ffma2(a2, make_float2(x.x, x.y), fmul2(k2, make_float2(u.x, u.y)));
    const float2 hi = ffma2(a2, make_float2(x.z, x.w), fmul2(k2, make_float2(u.z, u.w)));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <int D, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 2)
kda_decode_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                  const uint16_t* __restrict__ v, const float* __restrict__ log_alpha,
                  const uint16_t* __restrict__ beta, float* __restrict__ state,
                  void* __restrict__ out, int out_f32)
{
    using Sh = DecodeShape<D, WARPS>;
    __shared__ __align__(16) float2 s_akq[D], s_ak2[D];   // (alpha k, alpha q) and (alpha, k) per row
    __shared__ float s_u[D];
    __shared__ float s_red[WARPS][2][D];
    __shared__ float s_qk[WARPS];

    const int pair = blockIdx.x;                       // n * H + h
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float4* S = reinterpret_cast<float4*>(state + static_cast<size_t>(pair) * D * D);

    // 1. put the whole slice of the state this thread owns in flight
    const int c4 = lane % Sh::kLanesPerRow;
    const int rsub = lane / Sh::kLanesPerRow;
    float4 s[Sh::kIters];
#pragma unroll
    for (int it = 0; it < Sh::kIters; ++it) {
        const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
        s[it] = __ldcs(S + r * Sh::kLanesPerRow + c4);
    }

    // 2. per-row scalars: alpha, alpha*k, alpha*q, and q . k
    float qk_part = 0.f;
    if (tid < D) {
        const size_t o = static_cast<size_t>(pair) * D + tid;
        const float qi = bf16_bits_to_f32(q[o]);
        const float ki = bf16_bits_to_f32(k[o]);
        const float a = expf(log_alpha[o]);
        s_ak2[tid] = make_float2(a, ki);
        s_akq[tid] = make_float2(a * ki, a * qi);
        qk_part = qi * ki;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) qk_part += __shfl_xor_sync(0xffffffffu, qk_part, off);
    if (lane == 0) s_qk[warp] = qk_part;
    __syncthreads();

    // 3. partial column sums of S'^T k and S'^T q over this thread's rows
    float4 r1 = make_float4(0.f, 0.f, 0.f, 0.f), r2 = r1;
#pragma unroll
    for (int it = 0; it < Sh::kIters; ++it) {
        const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
        const float2 akq = s_akq[r];
        const float ak = akq.x, aq = akq.y;
        col_sums(r1, r2, ak, aq, s[it]);
    }
#pragma unroll
    for (int off = Sh::kLanesPerRow; off < 32; off <<= 1) {
        r1.x += __shfl_xor_sync(0xffffffffu, r1.x, off); r1.y += __shfl_xor_sync(0xffffffffu, r1.y, off);
        r1.z += __shfl_xor_sync(0xffffffffu, r1.z, off); r1.w += __shfl_xor_sync(0xffffffffu, r1.w, off);
        r2.x += __shfl_xor_sync(0xffffffffu, r2.x, off); r2.y += __shfl_xor_sync(0xffffffffu, r2.y, off);
        r2.z += __shfl_xor_sync(0xffffffffu, r2.z, off); r2.w += __shfl_xor_sync(0xffffffffu, r2.w, off);
    }
    if (rsub == 0) {
        *reinterpret_cast<float4*>(&s_red[warp][0][4 * c4]) = r1;
        *reinterpret_cast<float4*>(&s_red[warp][1][4 * c4]) = r2;
    }
    __syncthreads();

    // 4. finish the reductions: u = v - S'^T k, o = S'^T q + beta (q.k) u
    const float b = bf16_bits_to_f32(beta[pair]);
    if (tid < D) {
        float t1 = 0.f, t2 = 0.f, qk = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) { t1 += s_red[w][0][tid]; t2 += s_red[w][1][tid]; qk += s_qk[w]; }
        const size_t o = static_cast<size_t>(pair) * D + tid;
        const float u = bf16_bits_to_f32(v[o]) - t1;
        s_u[tid] = u;
        const float ov = t2 + b * qk * u;
        if (out_f32) reinterpret_cast<float*>(out)[o] = ov;
        else reinterpret_cast<uint16_t*>(out)[o] = f32_to_bf16_bits(ov);
    }
    __syncthreads();

    // 5. S = Diag(alpha) S + beta k u^T, written back in place
    const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * c4]);
#pragma unroll
    for (int it = 0; it < Sh::kIters; ++it) {
        const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
        const float2 ak2 = s_ak2[r];
        const float a = ak2.x;
        const float kr = b * ak2.y;
        __stcs(S + r * Sh::kLanesPerRow + c4, state_update(s[it], a, kr, u4));
    }
}

// ---------------------------------------------------------------------------------------
// Serving-shaped decode (pages: the DSpark speculative decoding of the serving notes, and
// the prefix-cache state pool of section 5).  Sequence n's state lives in slot
// slots[n] of a state pool; up to K of its tokens are applied in one pass: the state is
// read once, stepped K times in registers (each step exactly the single-token update
// above), and written back once -- or not at all (verify: outputs only, the pool is left
// untouched so the caller can accept any prefix and commit it with a second call).
// ---------------------------------------------------------------------------------------
constexpr int kStatusBadIndex = -1;     // KDA_ERR_INVALID_ARG, recorded on the device

template <int D, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 2)
kda_decode_multi_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                        const uint16_t* __restrict__ v, const float* __restrict__ log_alpha,
                        const uint16_t* __restrict__ beta, float* __restrict__ pool, int num_slots,
                        const int32_t* __restrict__ slots, const int32_t* __restrict__ ntok, int commit,
                        void* __restrict__ out, int out_f32, int K, int H, int decay, int* status)
{
    using Sh = DecodeShape<D, WARPS>;
    // per-row scalars of a token, double-buffered by token parity so that the next token's
    // may be written while slower warps still read this one's: (alpha k, alpha q), (alpha, k)
    __shared__ __align__(16) float2 s_akq[2][D], s_ak2[2][D];
    __shared__ float s_u[D];
    __shared__ float s_red[WARPS][2][D];
    __shared__ float s_qk[2][WARPS];

    const int pair = blockIdx.x;                       // n * H + h
    const int n = pair / H, h = pair - n * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = slots ? slots[n] : n;
    const int nt = ntok ? ntok[n] : K;
    if (slot < 0 || slot >= num_slots || nt < 0 || nt > K) {
        if (tid == 0) set_status(status, kStatusBadIndex);
        return;
    }
    float4* S = reinterpret_cast<float4*>(pool + (static_cast<size_t>(slot) * H + h) * D * D);

    const int c4 = lane % Sh::kLanesPerRow;
    const int rsub = lane / Sh::kLanesPerRow;
    float4 s[Sh::kIters];
#pragma unroll
    for (int it = 0; it < Sh::kIters; ++it) {
        const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
        s[it] = commit ? __ldcs(S + r * Sh::kLanesPerRow + c4) : __ldg(S + r * Sh::kLanesPerRow + c4);
    }

    // Token inputs (row tid of q, k, v, log_alpha, and beta) are fetched one token ahead, so
    // no token waits on a global load between its barriers.
    uint16_t q_in = 0, k_in = 0, v_in = 0, b_in = 0;
    float la_in = 0.f;
    auto fetch = [&](int j) {
        const size_t tok = static_cast<size_t>(n) * K + j;          // token row [n][j]
        const size_t vec = (tok * H + h) * D;                       // its [H, D] vectors
        if (tid < D) {
            q_in = q[vec + tid];
            k_in = k[vec + tid];
            v_in = v[vec + tid];
            // decay layouts: per channel (KDA), per head (Gated DeltaNet), none (DeltaNet)
            la_in = decay == 0 ? log_alpha[vec + tid] : decay == 1 ? log_alpha[tok * H + h] : 0.f;
        }
        b_in = beta[tok * H + h];
    };
    if (nt > 0) fetch(0);
    for (int j = 0; j < nt; ++j) {
        const size_t tok = static_cast<size_t>(n) * K + j;          // token row [n][j]
        const size_t vec = (tok * H + h) * D;                       // its [H, D] vectors
        const uint16_t q_j = q_in, k_j = k_in, v_j = v_in, b_j = b_in;
        const float la_j = la_in;
        if (j + 1 < nt) fetch(j + 1);
        float qk_part = 0.f;
        if (tid < D) {
            const float qi = bf16_bits_to_f32(q_j);
            const float ki = bf16_bits_to_f32(k_j);
            const float a = decay == 2 ? 1.f : expf(la_j);
            s_ak2[j & 1][tid] = make_float2(a, ki);
            s_akq[j & 1][tid] = make_float2(a * ki, a * qi);
            qk_part = qi * ki;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) qk_part += __shfl_xor_sync(0xffffffffu, qk_part, off);
        if (lane == 0) s_qk[j & 1][warp] = qk_part;
        __syncthreads();

        float4 r1 = make_float4(0.f, 0.f, 0.f, 0.f), r2 = r1;
#pragma unroll
        for (int it = 0; it < Sh::kIters; ++it) {
            const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
            const float2 akq = s_akq[j & 1][r];
        const float ak = akq.x, aq = akq.y;
            col_sums(r1, r2, ak, aq, s[it]);
        }
#pragma unroll
        for (int off = Sh::kLanesPerRow; off < 32; off <<= 1) {
            r1.x += __shfl_xor_sync(0xffffffffu, r1.x, off); r1.y += __shfl_xor_sync(0xffffffffu, r1.y, off);
            r1.z += __shfl_xor_sync(0xffffffffu, r1.z, off); r1.w += __shfl_xor_sync(0xffffffffu, r1.w, off);
            r2.x += __shfl_xor_sync(0xffffffffu, r2.x, off); r2.y += __shfl_xor_sync(0xffffffffu, r2.y, off);
            r2.z += __shfl_xor_sync(0xffffffffu, r2.z, off); r2.w += __shfl_xor_sync(0xffffffffu, r2.w, off);
        }
        if (rsub == 0) {
            *reinterpret_cast<float4*>(&s_red[warp][0][4 * c4]) = r1;
            *reinterpret_cast<float4*>(&s_red[warp][1][4 * c4]) = r2;
        }
        __syncthreads();

        const float b = bf16_bits_to_f32(b_j);
        if (tid < D) {
            float t1 = 0.f, t2 = 0.f, qk = 0.f;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) { t1 += s_red[w][0][tid]; t2 += s_red[w][1][tid]; qk += s_qk[j & 1][w]; }
            const float u = bf16_bits_to_f32(v_j) - t1;
            s_u[tid] = u;
            const float ov = t2 + b * qk * u;
            if (out_f32) reinterpret_cast<float*>(out)[vec + tid] = ov;
            else reinterpret_cast<uint16_t*>(out)[vec + tid] = f32_to_bf16_bits(ov);
        }
        __syncthreads();

        const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * c4]);
#pragma unroll
        for (int it = 0; it < Sh::kIters; ++it) {
            const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
            const float2 ak2 = s_ak2[j & 1][r];
            const float a = ak2.x;
            const float kr = b * ak2.y;
            s[it] = state_update(s[it], a, kr, u4);
        }
        // (no barrier here: the next token stages its scalars in the other buffer, and s_u and
        // s_red are next written only after the next token's first barrier, which every
        // thread reaches only when done with this token)
    }
    if (commit && nt > 0) {
#pragma unroll
        for (int it = 0; it < Sh::kIters; ++it) {
            const int r = warp * Sh::kRowsPerWarp + it * Sh::kRowsPerIter + rsub;
            __stcs(S + r * Sh::kLanesPerRow + c4, s[it]);
        }
    }
}

int launch_decode_multi(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                        const uint16_t* beta, float* pool, int num_slots, const int32_t* slots,
                        const int32_t* ntok, int commit, void* out, int out_f32,
                        int N, int K, int H, int D, int decay, int* status, cudaStream_t stream)
{
    const long long pairs = static_cast<long long>(N) * H;
    if (pairs == 0) return 0;
    if (D == 128) {
        kda_decode_multi_kernel<128, 8><<<static_cast<unsigned>(pairs), 256, 0, stream>>>(
            q, k, v, log_alpha, beta, pool, num_slots, slots, ntok, commit, out, out_f32, K, H, decay, status);
    } else {
        kda_decode_multi_kernel<64, 4><<<static_cast<unsigned>(pairs), 128, 0, stream>>>(
            q, k, v, log_alpha, beta, pool, num_slots, slots, ntok, commit, out, out_f32, K, H, decay, status);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                  const uint16_t* beta, float* state, void* out, int out_f32,
                  int N, int H, int D, cudaStream_t stream)
{
    const int pairs = N * H;
    if (pairs == 0) return 0;
    if (D == 128) {
        kda_decode_kernel<128, 8><<<pairs, 256, 0, stream>>>(q, k, v, log_alpha, beta, state, out, out_f32);
    } else {
        kda_decode_kernel<64, 4><<<pairs, 128, 0, stream>>>(q, k, v, log_alpha, beta, state, out, out_f32);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace kda
