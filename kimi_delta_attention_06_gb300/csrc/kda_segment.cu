// kda_segment.cu -- device helpers of the segmented prefill (kda_chunk_prefill_segmented).
//
// The KDA recurrence S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
// (Kimi Linear, "Kimi Delta Attention", the per-channel gated delta rule) is linear in the
// pair (S_0, v): over a segment of tokens, S_end = Phi S_0 + B, where Phi (Dk x Dk) is the
// product of the segment's per-token transitions and B is the state the segment reaches
// from S_0 = 0.  The prefill kernel itself yields both: B is the final state of a run from
// zeros, and Phi the final state of a run from S_0 = I with v = 0.  The helpers here set
// up those runs (segment bounds, identity and zero initial states) and chain the segment
// results: S_start[p + 1] = Phi_p S_start[p] + B_p, serially over the segments.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kda {

namespace {

// The runs' index arrays (built on the host), then their initial states: ident
// [n_ident, H, D, D] = I per head; zinit [n_zinit, H, D, D] = the prompt's initial state in
// slot 0 (zeros if none) and zeros elsewhere.
__global__ void seg_setup_kernel(SegIdxBuf ib, int32_t* idx, float* ident, int n_ident, float* zinit, int n_zinit,
                                 const float* init_state, int H, int D) {
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nth = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = tid; e < ib.n; e += nth) idx[e] = ib.v[e];
    const long long per = static_cast<long long>(H) * D * D;                           // one state slot
    for (long long e = tid; e < static_cast<long long>(n_ident) * per; e += nth) {
        const int rc = static_cast<int>(e % (static_cast<long long>(D) * D));
        ident[e] = (rc / D == rc % D) ? 1.f : 0.f;
    }
    for (long long e = tid; e < static_cast<long long>(n_zinit) * per; e += nth)
        zinit[e] = (e < per && init_state) ? init_state[e] : 0.f;
}

// Chain the segment results, one CTA per (16-column block, head): the state's columns are
// independent, so each CTA carries a Dk x 16 slab of S_start through the segments in order.
// phi   [P-2, H, D, D]  transitions of segments 1 .. P-2
// sst   [P, H, D, D]    slot 1 holds segment 0's final state; slot p + 1 (p = 1 .. P-2) holds
//                       B_p on entry and S_start[p + 1] = Phi_p S_start[p] + B_p on exit
// (slot 0, the prompt's own initial state, is not touched)
__global__ void __launch_bounds__(256) seg_chain_kernel(const float* __restrict__ phi, float* sst, int P, int H,
                                                         int D) {
    __shared__ __align__(16) float slab[128][16];
    const int h = blockIdx.y, c0 = 16 * blockIdx.x;
    const int i = threadIdx.x >> 1, j0 = 8 * (threadIdx.x & 1);     // row, first of 8 columns
    const size_t per = static_cast<size_t>(H) * D * D;
    const size_t head = static_cast<size_t>(h) * D * D;
    if (i < D) {
        const float* s1 = sst + per + head + static_cast<size_t>(i) * D + c0 + j0;
#pragma unroll
        for (int j = 0; j < 8; ++j) slab[i][j0 + j] = s1[j];
    }
    __syncthreads();
    for (int p = 1; p <= P - 2; ++p) {
        float acc[8];
        float* dst = sst + static_cast<size_t>(p + 1) * per + head + static_cast<size_t>(i) * D + c0 + j0;
        if (i < D) {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = dst[j];                // B_p
            const float* row = phi + static_cast<size_t>(p - 1) * per + head + static_cast<size_t>(i) * D;
            for (int kk = 0; kk < D; kk += 4) {
                const float4 f = *reinterpret_cast<const float4*>(row + kk);
                const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = fmaf(fv[u], slab[kk + u][j0 + j], acc[j]);
                }
            }
        }
        __syncthreads();                                                // every row has read the slab
        if (i < D) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                slab[i][j0 + j] = acc[j];
                dst[j] = acc[j];
            }
        }
        __syncthreads();
    }
}

}  // namespace

int launch_segment_setup(const SegIdxBuf& ib, int32_t* idx, float* ident, int n_ident, float* zinit, int n_zinit,
                         const float* init_state, int H, int D, cudaStream_t stream) {
    if (ib.n < 0 || ib.n > kSegIdxMax || n_ident < 0 || n_zinit < 0) return -1;
    seg_setup_kernel<<<4 * 152, 256, 0, stream>>>(ib, idx, ident, n_ident, zinit, n_zinit, init_state, H, D);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_segment_chain(const float* phi, float* sst, int P, int H, int D, cudaStream_t stream) {
    if (P < 3 || (D != 64 && D != 128)) return -1;
    const dim3 grid(D / 16, H);
    seg_chain_kernel<<<grid, 256, 0, stream>>>(phi, sst, P, H, D);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace kda
