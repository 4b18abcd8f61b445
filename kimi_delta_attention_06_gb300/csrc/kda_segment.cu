// kda_segment.cu -- device helpers of the segmented prefill (kda_chunk_prefill_segmented_ex).
//
// The KDA recurrence S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
// (Kimi Linear, "Kimi Delta Attention", the per-channel gated delta rule) is linear in the
// pair (S_0, v): over a segment of tokens, S_end = Phi S_0 + B, where Phi (Dk x Dk) is the
// product of the segment's per-token transitions and B is the state the segment reaches
// from S_0 = 0.  The prefill kernel itself yields both: B is the final state of a run from
// zeros, and Phi the final state of a run from S_0 = I with v = 0.  Each sequence of a call
// is cut into segments; three prefill launches run over the list of all segments, each with
// a skip list that picks the segments it forms (A: B_p and the first segment's true end
// state; B: Phi_p; F: the outputs from the chained start states).  The helpers here set up
// those runs and chain the segment results of each sequence serially:
// S_start[p + 1] = Phi_p S_start[p] + B_p.
//
// A transition that cannot matter is not formed.  Each token's factor has spectral norm at
// most max_c alpha_{t,c} * max(1, |1 - beta_t |k_t|^2|) (the projection I - beta k k^T has
// eigenvalues 1 and 1 - beta |k|^2), so log ||Phi_p|| <= sum over the segment of
// max_c log alpha_{t,c} + log max(1, |1 - beta_t |k_t|^2|).  Where that bound is below
// kSkipLogNorm (2^-64, far under fp32 rounding of the state), Phi_p S_start[p] is dropped:
// its run is skipped and S_start[p + 1] = B_p.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kda {

namespace {

constexpr float kSkipLogNorm = -44.3614195558365f;   // -64 ln 2
constexpr int kBoundBlocks = kSegBoundBlocks;

// Segment roles (bits of the role array): first / last segment of its sequence, and whether
// the sequence is split at all (a sequence of one segment runs as a plain prefill in run F).
__device__ __forceinline__ bool runs_in_a(int r) { return (r & kSegMulti) && !(r & kSegLast); }
__device__ __forceinline__ bool runs_in_b(int r) { return (r & kSegMulti) && !(r & (kSegFirst | kSegLast)); }
__device__ __forceinline__ bool runs_in_f(int r) { return !(r & kSegMulti) || !(r & kSegFirst); }

// Copies the index arrays (built on the host) to the device, then per segment g:
//   ident[g] = I;  zin[g] = the sequence's initial state if g is its first segment, else 0
//   (run A's initial states);  sst[g] = the sequence's initial state if g is its first
//   segment (run F's initial state of an unsplit sequence; run A and the chain fill the
//   others);  skip_a / skip_f = whether runs A / F leave the segment out (per head).
__global__ void seg_setup_kernel(SegIdxBuf ib, int32_t* idx, int n_seg, int o_role, int o_seq, int H, int D,
                                 const float* init_state, float* ident, float* zin, float* sst, int* skip_a,
                                 int* skip_f) {
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nth = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = tid; e < ib.n; e += nth) idx[e] = ib.v[e];
    for (long long e = tid; e < static_cast<long long>(n_seg) * H; e += nth) {
        const int r = ib.v[o_role + e / H];
        skip_a[e] = runs_in_a(r) ? 0 : 1;
        skip_f[e] = runs_in_f(r) ? 0 : 1;
    }
    const long long per = static_cast<long long>(H) * D * D;                           // one state slot
    for (long long e = tid; e < static_cast<long long>(n_seg) * per; e += nth) {
        const int g = static_cast<int>(e / per);
        const long long w = e % per;
        const int rc = static_cast<int>(w % (static_cast<long long>(D) * D));
        ident[e] = (rc / D == rc % D) ? 1.f : 0.f;
        const bool first = (ib.v[o_role + g] & kSegFirst) != 0;
        const float s0 = (first && init_state) ? init_state[static_cast<long long>(ib.v[o_seq + g]) * per + w] : 0.f;
        zin[e] = s0;
        if (first) sst[e] = s0;
    }
}

// Partial sums of the bound above: grid (kBoundBlocks, segments, H), one warp per token
// (lanes over channels), warps and blocks strided over the segment's tokens; segments that
// run B leaves out are not read.  seg_cu [n_seg + 1]: token bounds of the segments;
// partial [(seg * H + h) * kBoundBlocks + blk].
__global__ void __launch_bounds__(256) seg_bound_kernel(const uint16_t* __restrict__ k, const float* __restrict__ la,
                                                        const uint16_t* __restrict__ beta, int decay, int H, int D,
                                                        const int32_t* __restrict__ seg_cu,
                                                        const int32_t* __restrict__ role, float* partial) {
    __shared__ float s_w[8];
    const int blk = blockIdx.x, seg = blockIdx.y, h = blockIdx.z;
    if (!runs_in_b(role[seg])) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = seg_cu[seg], t1 = seg_cu[seg + 1];
    const bool lane_ok = 4 * lane < D;
    float acc = 0.f;
    for (int t = t0 + blk * 8 + warp; t < t1; t += 8 * kBoundBlocks) {
        const size_t row = static_cast<size_t>(t) * H + h;
        float m = 0.f, kk = 0.f;
        if (lane_ok) {
            const uint2 kw = *reinterpret_cast<const uint2*>(k + row * D + 4 * lane);
            const float2 k01 = bf16x2_bits_to_f32(kw.x), k23 = bf16x2_bits_to_f32(kw.y);
            kk = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
        }
        if (decay == 0) {          // per channel: the largest log-decay of the token
            m = -INFINITY;
            if (lane_ok) {
                const float4 a = *reinterpret_cast<const float4*>(la + row * D + 4 * lane);
                m = fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, o);
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        }
        if (decay == 1) m = la[row];
        const float b = bf16_bits_to_f32(beta[row]);
        acc += m + logf(fmaxf(1.f, fabsf(1.f - b * kk)));
    }
    if (lane == 0) s_w[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float sum = 0.f;
        for (int w = 0; w < 8; ++w) sum += s_w[w];
        partial[(static_cast<size_t>(seg) * H + h) * kBoundBlocks + blk] = sum;
    }
}

// Run B's skip list: segments it does not form, and those whose transition the bound rules
// out (decay 2, none, rules out nothing).
__global__ void seg_flag_kernel(const float* partial, const int32_t* role, int n_seg, int H, int decay, int* skip_b) {
    for (int i = threadIdx.x; i < n_seg * H; i += blockDim.x) {
        const int g = i / H;
        int sk = 1;
        if (runs_in_b(role[g])) {
            sk = 0;
            if (decay != 2) {
                const float* pp = partial + static_cast<size_t>(i) * kBoundBlocks;
                float sum = 0.f;
                for (int b = 0; b < kBoundBlocks; ++b) sum += pp[b];
                sk = sum < kSkipLogNorm ? 1 : 0;
            }
        }
        skip_b[i] = sk;
    }
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kSlab = 4;          // state columns per CTA

// Chain the segment results of each split sequence, one CTA per (4-column block, head,
// sequence): the state's columns are independent, so each CTA carries a D x 4 slab of its
// sequence's S_start through the sequence's segments in order.  Each step's Phi (D x D,
// contiguous) is copied into shared memory (row pitch D + 4) while the previous step
// computes; thread (row i, columns 2 (tid & 1) .. +1) forms its two outputs as fp32 dot
// products over the whole row.  For chain z, segments g0 .. g0 + P - 1 (global indices):
// phi   [n_seg, H, D, D]  slot g holds Phi of segment g (formed where skip_b is 0)
// sst   [n_seg, H, D, D]  slot g0 + 1 holds the end state of segment g0; slot g0 + p + 1
//                         (p = 1 .. P-2) holds B on entry and S_start = Phi S_start + B on exit
__global__ void __launch_bounds__(256) seg_chain_kernel(SegChainBuf cb, const float* __restrict__ phi,
                                                         const int* __restrict__ skip_b, float* sst, int H, int D) {
    extern __shared__ __align__(16) float sm[];
    const int pitch = D + 4;
    float* slab = sm;                                 // [D][kSlab]
    float* phis = sm + 128 * kSlab;                   // 2 x [D][pitch]
    const int h = blockIdx.y, c0 = kSlab * blockIdx.x;
    const int g0 = cb.g0[blockIdx.z], P = cb.np[blockIdx.z];
    const int i = threadIdx.x >> 1, j0 = 2 * (threadIdx.x & 1);
    const size_t per = static_cast<size_t>(H) * D * D;
    const size_t head = static_cast<size_t>(h) * D * D;
    auto stage = [&](int p) {                         // Phi of segment g0 + p into buffer (p - 1) & 1
        const float* src = phi + static_cast<size_t>(g0 + p) * per + head;
        float* dst = phis + ((p - 1) & 1) * D * pitch;
        const int q4 = D / 4;
        for (int e = threadIdx.x; e < D * q4; e += blockDim.x) {
            const int r = e / q4, c = 4 * (e % q4);
            cp_async16(dst + r * pitch + c, src + static_cast<size_t>(r) * D + c);
        }
        cp_async_commit();
    };
    if (i < D) {
        const float* s1 = sst + static_cast<size_t>(g0 + 1) * per + head + static_cast<size_t>(i) * D + c0 + j0;
        slab[i * kSlab + j0] = s1[0];
        slab[i * kSlab + j0 + 1] = s1[1];
    }
    stage(1);
    for (int p = 1; p <= P - 2; ++p) {
        if (p + 1 <= P - 2) {
            stage(p + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();                              // Phi and the slab are in place
        float a0 = 0.f, a1 = 0.f;
        float* dst = sst + static_cast<size_t>(g0 + p + 1) * per + head +
                     static_cast<size_t>(i < D ? i : 0) * D + c0 + j0;
        const bool use_phi = !skip_b[static_cast<size_t>(g0 + p) * H + h];
        if (i < D) {
            a0 = dst[0];                              // B
            a1 = dst[1];
        }
        if (i < D && use_phi) {
            const float* row = phis + ((p - 1) & 1) * D * pitch + i * pitch;
#pragma unroll 8
            for (int kk = 0; kk < D; kk += 4) {
                const float4 f = *reinterpret_cast<const float4*>(row + kk);
                const float2 s0 = *reinterpret_cast<const float2*>(slab + (kk + 0) * kSlab + j0);
                const float2 s1 = *reinterpret_cast<const float2*>(slab + (kk + 1) * kSlab + j0);
                const float2 s2 = *reinterpret_cast<const float2*>(slab + (kk + 2) * kSlab + j0);
                const float2 s3 = *reinterpret_cast<const float2*>(slab + (kk + 3) * kSlab + j0);
                a0 = fmaf(f.x, s0.x, a0); a1 = fmaf(f.x, s0.y, a1);
                a0 = fmaf(f.y, s1.x, a0); a1 = fmaf(f.y, s1.y, a1);
                a0 = fmaf(f.z, s2.x, a0); a1 = fmaf(f.z, s2.y, a1);
                a0 = fmaf(f.w, s3.x, a0); a1 = fmaf(f.w, s3.y, a1);
            }
        }
        __syncthreads();                              // every row has read the slab and Phi
        if (i < D) {
            slab[i * kSlab + j0] = a0;
            slab[i * kSlab + j0 + 1] = a1;
            dst[0] = a0;
            dst[1] = a1;
        }
    }
}

}  // namespace

int launch_segment_setup(const SegIdxBuf& ib, int32_t* idx, int n_seg, int o_role, int o_seq, int H, int D,
                         const float* init_state, float* ident, float* zin, float* sst, int* skip_a, int* skip_f,
                         cudaStream_t stream) {
    if (ib.n < 0 || ib.n > kSegIdxMax || n_seg < 0 || o_role < 0 || o_seq < 0 || o_role + n_seg > ib.n ||
        o_seq + n_seg > ib.n)
        return -1;
    seg_setup_kernel<<<4 * 152, 256, 0, stream>>>(ib, idx, n_seg, o_role, o_seq, H, D, init_state, ident, zin, sst,
                                                  skip_a, skip_f);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_segment_bound(const uint16_t* k, const float* la, const uint16_t* beta, int decay, int H, int D,
                         const int32_t* seg_cu, const int32_t* role, int n_seg, float* partial, int* skip_b,
                         cudaStream_t stream) {
    if (n_seg <= 0 || H <= 0 || (D != 64 && D != 128) || decay < 0 || decay > 2) return -1;
    if (decay != 2) {
        const dim3 grid(kBoundBlocks, n_seg, H);
        seg_bound_kernel<<<grid, 256, 0, stream>>>(k, la, beta, decay, H, D, seg_cu, role, partial);
    }
    seg_flag_kernel<<<1, 256, 0, stream>>>(partial, role, n_seg, H, decay, skip_b);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_segment_chain(const SegChainBuf& cb, const float* phi, const int* skip_b, float* sst, int H, int D,
                         cudaStream_t stream) {
    if (cb.n <= 0 || cb.n > kSegMaxChains || (D != 64 && D != 128)) return -1;
    const int smem = static_cast<int>(sizeof(float) * (128 * kSlab + 2 * D * (D + 4)));
    static bool attr_done[kMaxDevicesAttr] = {};
    if (!raise_smem_limit(reinterpret_cast<const void*>(seg_chain_kernel), 128 * kSlab * 4 + 2 * 128 * 132 * 4,
                          attr_done))
        return -3;
    const dim3 grid(D / kSlab, H, cb.n);
    seg_chain_kernel<<<grid, 256, smem, stream>>>(cb, phi, skip_b, sst, H, D);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace kda
