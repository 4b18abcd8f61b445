// kda_api.cu -- the C ABI declared in include/kda.h: host-side validation,
// the device status word, and dispatch to the CUDA kernels.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>
#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "../../include/kda_debug.h"
#include "common.cuh"
#include "tc.cuh"

namespace kda {
int launch_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                  const uint16_t* beta, float* state, void* out, int out_f32,
                  int N, int H, int D, cudaStream_t stream);
int launch_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* la,
                   const uint16_t* beta, const float* init_state, const int32_t* cu_seqlens,
                   int num_seqs, int total_tokens, int H, int Dk, int Dv, void* out, int out_f32,
                   float* final_state, float* ckpt, int ckpt_stride, int decay, const int32_t* start_pos,
                   const float* norm_gamma, float norm_eps,
                   void* ws, int* ring_flags, int ring_count, int* status, cudaStream_t stream,
                   const int* skip = nullptr);
size_t prefill_workspace_bytes(int num_seqs, int H);
int prefill_ring_count(int num_seqs, int H);
int prefill_max_active_clusters();
int launch_prepare_inputs(const uint16_t* xq, const uint16_t* xk, const uint16_t* xv, const float* conv_w,
                          const uint16_t* conv_state, const float* a_raw, const uint16_t* b_raw,
                          const int32_t* cu_seqlens, int num_seqs, int T, int H, int D, int act,
                          uint16_t* q, uint16_t* k, uint16_t* v, float* log_alpha, uint16_t* beta,
                          int* status, cudaStream_t stream);
int launch_output_norm(const void* o, int o_f32, const float* gamma, float eps, uint16_t* y, int T, int H, int D,
                       cudaStream_t stream);
int launch_segment_setup(const SegIdxBuf& ib, int32_t* idx, int n_seg, int o_role, int o_seq, int H, int D,
                         const float* init_state, float* ident, float* zin, float* sst, int* skip_a, int* skip_f,
                         cudaStream_t stream);
int launch_segment_bound(const uint16_t* k, const float* la, const uint16_t* beta, int decay, int H, int D,
                         const int32_t* seg_cu, const int32_t* role, int n_seg, float* partial, int* skip_b,
                         cudaStream_t stream);
int launch_segment_chain(const SegChainBuf& cb, const float* phi, const int* skip_b, float* sst, int H, int D,
                         cudaStream_t stream);
int launch_decode_multi(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                        const uint16_t* beta, float* pool, int num_slots, const int32_t* slots,
                        const int32_t* ntok, int commit, void* out, int out_f32,
                        int N, int K, int H, int D, int decay, int* status, cudaStream_t stream);
}  // namespace kda

namespace {

// One status word per device (module-scope device variable; no allocation).
__device__ int g_kda_status = 0;

// Scratch of kda_chunk_prefill_noalloc: the hand-off rings of up to
// KDA_NOALLOC_MAX_SEQ_HEADS (sequence, head) pairs (module-scope, no allocation).
__device__ __align__(256) uint8_t g_kda_noalloc_scratch[KDA_NOALLOC_MAX_SEQ_HEADS * kda::kPrefillRingBytesPerPair];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
uint8_t* g_scratch_ptr[kMaxDevices] = {};
cudaMemPool_t g_pool[kMaxDevices] = {};   // stream-ordered pool for the prefill hand-off ring
int g_device_ok[kMaxDevices] = {};   // 0 unknown, 1 supported, -1 unsupported

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resolve the current device's status word (and fixed prefill scratch) and check
// it can run sm_103a code.
int device_setup(int** status, uint8_t** scratch = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return KDA_ERR_CUDA;
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_device_ok[dev] == 1) {
            void* p = nullptr;
            void* sp = nullptr;
            if (cudaGetSymbolAddress(&p, g_kda_status) != cudaSuccess ||
                cudaGetSymbolAddress(&sp, g_kda_noalloc_scratch) != cudaSuccess) {
                g_device_ok[dev] = 0;
                return KDA_ERR_CUDA;
            }
            g_status_ptr[dev] = static_cast<int*>(p);
            g_scratch_ptr[dev] = static_cast<uint8_t*>(sp);
        }
    }
    if (g_device_ok[dev] != 1) return KDA_ERR_UNSUPPORTED;
    *status = g_status_ptr[dev];
    if (scratch) *scratch = g_scratch_ptr[dev];
    return KDA_OK;
}

// The library's own memory pool on the current device (created once; it keeps what it
// has reserved, so steady-state calls reuse the same memory without a driver call).
int workspace_pool(cudaMemPool_t* pool) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pl = nullptr;
        if (cudaMemPoolCreate(&pl, &props) != cudaSuccess) return KDA_ERR_CUDA;
        uint64_t keep = ~0ull;
        if (cudaMemPoolSetAttribute(pl, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pl);
            return KDA_ERR_CUDA;
        }
        g_pool[dev] = pl;
    }
    *pool = g_pool[dev];
    return KDA_OK;
}

// A second stream per device for work that can run beside a prefill on the SMs it leaves idle
// (created once, non-blocking; ordered against the caller's stream with events).
cudaStream_t g_side[kMaxDevices] = {};
int side_stream(cudaStream_t* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_side[dev] && cudaStreamCreateWithFlags(&g_side[dev], cudaStreamNonBlocking) != cudaSuccess) {
        g_side[dev] = nullptr;
        return KDA_ERR_CUDA;
    }
    *out = g_side[dev];
    return KDA_OK;
}

bool head_dims_ok(int Dk, int Dv) { return (Dk == 64 || Dk == 128) && (Dv == 64 || Dv == 128); }

// Host-side checks shared by the two prefill entry points.
int check_prefill_args(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                       const uint16_t* beta, const float* init_state, const int32_t* cu_seqlens,
                       const int32_t* cu_seqlens_host, int num_seqs, int total_tokens, int H, int Dk, int Dv,
                       const void* out, int out_dtype, const float* final_state, const float* ckpt_states,
                       int ckpt_stride, int decay) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (decay != KDA_DECAY_CHANNEL && decay != KDA_DECAY_HEAD && decay != KDA_DECAY_NONE) return KDA_ERR_INVALID_ARG;
    if (decay == KDA_DECAY_HEAD && H % 4 != 0) return KDA_ERR_UNSUPPORTED;
    if (decay == KDA_DECAY_NONE && log_alpha) return KDA_ERR_INVALID_ARG;
    if (out_dtype != KDA_OUT_BF16 && out_dtype != KDA_OUT_F32) return KDA_ERR_INVALID_ARG;
    if (ckpt_stride < 0 || (ckpt_stride % 64) != 0) return KDA_ERR_INVALID_ARG;
    if (!head_dims_ok(Dk, Dv)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs > 0 && (!cu_seqlens || !cu_seqlens_host)) return KDA_ERR_INVALID_ARG;
    if (num_seqs > 0) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
        for (int n = 0; n < num_seqs; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
    } else if (total_tokens != 0) {
        return KDA_ERR_INVALID_ARG;
    }
    if (total_tokens > 0 && (!q || !k || !v || !beta || !out)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && decay != KDA_DECAY_NONE && !log_alpha) return KDA_ERR_INVALID_ARG;
    if (ckpt_states && ckpt_stride == 0) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, log_alpha, beta, init_state, out, final_state, ckpt_states, cu_seqlens};
    for (const void* p : ptrs)
        if (p && !aligned16(p) && p != cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return KDA_ERR_INVALID_ARG;
    // 32-bit element offsets inside the kernel stay below 2^31 per row of work
    if (static_cast<int64_t>(total_tokens) * H * (Dk > Dv ? Dk : Dv) >= (int64_t(1) << 40)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

// One thread waits, with a bound, on an mbarrier phase that nothing completes.
__global__ void expire_wait_kernel(unsigned long long limit_ns, int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        kda::tc::mbar_init(&bar, 1);
        kda::tc::mbar_fence_init();
        if (!kda::tc::mbar_wait_bounded(&bar, 0, limit_ns)) kda::set_status(status, kda::kStatusTimeout);
    }
}

// The plan of a segmented prefill over N sequences.  Every sequence of more than a few
// chunks is cut, on its absolute 64-token chunk grid, into P_n >= 3 segments of about L
// chunks (L = the call's chunks / `segments`, so that every run holds about `segments`
// segments per head); the others stay whole (P_n = 1).  All segments, in sequence order,
// tile the call's tokens, and each of the runs A, B and F covers all of them with a skip
// list.  Checkpoints: runs A and F write the same slot layout (per segment, the stride
// multiples strictly inside it, then its end; a skipped segment's slots stay unwritten);
// keep[i] is the slot, counted over run A's slots then run F's, of the call's i-th own
// checkpoint (a split sequence's first segment from run A, the rest from run F).
struct SegPlan {
    int n_seg = 0;
    std::vector<int32_t> cu, sp, role, seq;     // per segment (cu: n_seg + 1 bounds)
    std::vector<int32_t> g0, np;                // per split sequence: first segment, segments
    std::vector<int32_t> last;                  // per sequence: its last segment
    std::vector<int> keep;
    int64_t n_ck = 0;
};

constexpr int kSegMaxSeqs = 32;

int plan_segments(const int32_t* cu_host, const int32_t* sp_host, int N, int segments, int ckpt_stride,
                  SegPlan* out) {
    if (segments < 1 || segments > KDA_MAX_SEGMENTS || N < 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_stride < 0 || ckpt_stride % 64 != 0) return KDA_ERR_INVALID_ARG;
    if (N > 0 && !cu_host) return KDA_ERR_INVALID_ARG;
    const int C = 64;
    std::vector<int64_t> chunks(N);
    int64_t total = 0;
    for (int n = 0; n < N; ++n) {
        const int64_t len = static_cast<int64_t>(cu_host[n + 1]) - cu_host[n];
        const int64_t s0 = sp_host ? sp_host[n] : 0;
        if (len < 0 || s0 < 0 || s0 + len > INT32_MAX) return KDA_ERR_INVALID_ARG;
        chunks[n] = len > 0 ? (s0 + len + C - 1) / C - s0 / C : 0;
        total += chunks[n];
    }
    // segment length in chunks.  A sequence of one such segment stays whole; one of two is cut
    // too when the call has several sequences (its halves then sit in runs A and F, which
    // shortens the longest chain of each run), but not alone (two halves in series take as
    // long as the whole)
    const bool split_any = segments >= 3 && N <= kSegMaxSeqs && total >= 2;
    const int64_t L = split_any ? (total + segments - 1) / segments : 0;
    SegPlan pl;
    pl.cu.push_back(0);
    for (int n = 0; n < N; ++n) {
        const int64_t t0 = cu_host[n], len = static_cast<int64_t>(cu_host[n + 1]) - t0;
        const int64_t s0 = sp_host ? sp_host[n] : 0;
        int P = 1;
        if (split_any && chunks[n] >= 2) {
            P = static_cast<int>((chunks[n] + L - 1) / L);
            if (P < 2 || (N == 1 && P < 3)) P = 1;
        }
        if (P > 1 && static_cast<int>(pl.g0.size()) >= kda::kSegMaxChains) P = 1;
        const int g_first = pl.n_seg;
        for (int p = 0; p < P; ++p) {
            int64_t e = len;
            if (p + 1 < P) {
                const int64_t x = C * (s0 / C + (p + 1) * L) - s0;
                e = x < 0 ? 0 : (x > len ? len : x);
            }
            const int64_t a = pl.cu.back() - t0;
            pl.cu.push_back(static_cast<int32_t>(t0 + e));
            pl.sp.push_back(static_cast<int32_t>(s0 + a));
            int r = 0;
            if (p == 0) r |= kda::kSegFirst;
            if (p == P - 1) r |= kda::kSegLast;
            if (P > 1) r |= kda::kSegMulti;
            pl.role.push_back(r);
            pl.seq.push_back(n);
            ++pl.n_seg;
        }
        if (P > 1) { pl.g0.push_back(g_first); pl.np.push_back(P); }
        pl.last.push_back(pl.n_seg - 1);
    }
    if (ckpt_stride > 0) {
        // slot layout per segment, then which slots are the call's own checkpoints
        std::vector<int64_t> base(pl.n_seg + 1, 0);
        for (int g = 0; g < pl.n_seg; ++g) {
            const int64_t a = pl.sp[g], e = a + (pl.cu[g + 1] - pl.cu[g]);
            base[g + 1] = base[g] + (e > a ? (e - 1) / ckpt_stride - a / ckpt_stride + 1 : 0);
        }
        pl.n_ck = base[pl.n_seg];
        for (int g = 0; g < pl.n_seg; ++g) {
            const int64_t a = pl.sp[g], e = a + (pl.cu[g + 1] - pl.cu[g]);
            if (e <= a) continue;
            const bool from_a = (pl.role[g] & kda::kSegMulti) && (pl.role[g] & kda::kSegFirst);
            const int64_t off = from_a ? 0 : pl.n_ck;
            int64_t s = base[g];
            for (int64_t m = (a / ckpt_stride + 1) * ckpt_stride; m < e; m += ckpt_stride)
                pl.keep.push_back(static_cast<int>(off + s++));
            if (e % ckpt_stride == 0 || (pl.role[g] & kda::kSegLast)) pl.keep.push_back(static_cast<int>(off + s));
        }
        if (static_cast<int64_t>(pl.keep.size()) != kda_ckpt_count_ex(cu_host, sp_host, N, ckpt_stride))
            return KDA_ERR_INVALID_ARG;
    }
    *out = std::move(pl);
    return KDA_OK;
}

}  // namespace

extern "C" {

int64_t kda_ckpt_count_ex(const int32_t* cu_seqlens_host, const int32_t* start_pos_host, int num_seqs,
                          int ckpt_stride) {
    if (num_seqs < 0 || ckpt_stride < 0 || (num_seqs > 0 && !cu_seqlens_host)) return -1;
    if (ckpt_stride == 0) return 0;
    int64_t total = 0;
    for (int n = 0; n < num_seqs; ++n) {
        const int64_t len = static_cast<int64_t>(cu_seqlens_host[n + 1]) - cu_seqlens_host[n];
        const int64_t s = start_pos_host ? start_pos_host[n] : 0;
        if (len < 0 || s < 0) return -1;
        // stride multiples strictly inside (s, s + len), plus the end
        if (len > 0) total += (s + len - 1) / ckpt_stride - s / ckpt_stride + 1;
    }
    return total;
}

int64_t kda_ckpt_count(const int32_t* cu_seqlens_host, int num_seqs, int ckpt_stride) {
    return kda_ckpt_count_ex(cu_seqlens_host, nullptr, num_seqs, ckpt_stride);
}

int kda_chunk_size(void) { return 64; }

int kda_segment_plan(int total_tokens, int start_pos, int segments, int ckpt_stride, int32_t* bounds,
                     int32_t* ckpt_slots, int ckpt_slots_cap) {
    if (!bounds || total_tokens < 0 || start_pos < 0) return KDA_ERR_INVALID_ARG;
    const int32_t cu1[2] = {0, total_tokens};
    const int32_t sp1[1] = {start_pos};
    SegPlan plan;
    const int rc = plan_segments(cu1, sp1, 1, segments, ckpt_stride, &plan);
    if (rc != KDA_OK) return rc;
    const bool split = plan.n_seg > 1;
    if (ckpt_slots && split && static_cast<int64_t>(plan.keep.size()) > ckpt_slots_cap) return KDA_ERR_INVALID_ARG;
    for (int g = 0; g <= plan.n_seg; ++g) bounds[g] = plan.cu[g];
    if (ckpt_slots && split)
        for (size_t i = 0; i < plan.keep.size(); ++i) ckpt_slots[i] = plan.keep[i];
    return plan.n_seg;
}

int kda_prefill_clusters_at_once(void) {
    int* status = nullptr;
    const int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    const int n = kda::prefill_max_active_clusters();
    return n > 0 ? n : KDA_ERR_CUDA;
}

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape or device";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_TIMEOUT: return "device-side wait timed out";
        case KDA_ERR_RANGE: return "input outside the prefill's numeric domain";
        default: return "unknown status";
    }
}

static int prefill_pooled(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* log_alpha,
                          const uint16_t* beta, const float* init_state, const int32_t* cu_seqlens,
                          const int32_t* cu_seqlens_host, int num_seqs, int total_tokens, int H, int Dk, int Dv,
                          void* out, int out_dtype, float* final_state, float* ckpt_states, int ckpt_stride,
                          int decay, const int32_t* start_pos, const int32_t* start_pos_host,
                          const float* norm_gamma, float norm_eps, void* stream, const int* skip = nullptr) {
    int rc = check_prefill_args(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host, num_seqs,
                                total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, decay);
    if (rc != KDA_OK || num_seqs == 0) return rc;
    if (norm_gamma && (!aligned16(norm_gamma) || !(norm_eps >= 0.f) || !(norm_eps < 3.0e38f))) return KDA_ERR_INVALID_ARG;
    if ((start_pos == nullptr) != (start_pos_host == nullptr)) return KDA_ERR_INVALID_ARG;
    if (start_pos) {
        if (reinterpret_cast<uintptr_t>(start_pos) & 3u) return KDA_ERR_INVALID_ARG;
        for (int n = 0; n < num_seqs; ++n)
            if (start_pos_host[n] < 0) return KDA_ERR_INVALID_ARG;
    }
    int* status = nullptr;
    rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(&pool);
    if (rc != KDA_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    // rings for the clusters that can run at once (claimed per cluster), then their flags
    const int rings = kda::prefill_ring_count(num_seqs, H);
    if (rings <= 0) return KDA_ERR_CUDA;
    const size_t ring_bytes = kda::prefill_workspace_bytes(1, rings);
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, ring_bytes + sizeof(int) * rings, pool, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    int* flags = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ring_bytes);
    rc = kda::launch_prefill(q, k, v, log_alpha, beta, init_state, cu_seqlens, num_seqs, total_tokens, H, Dk, Dv,
                             out, out_dtype == KDA_OUT_F32, final_state, ckpt_states, ckpt_stride, decay,
                             start_pos, norm_gamma, norm_eps, ws, flags, rings, status, st, skip);
    const bool freed = cudaFreeAsync(ws, st) == cudaSuccess;
    return (rc == 0 && freed) ? KDA_OK : KDA_ERR_CUDA;
}

int kda_chunk_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const float* log_alpha, const uint16_t* beta,
                      const float* init_state,
                      const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                      int num_seqs, int total_tokens, int H, int Dk, int Dv,
                      void* out, int out_dtype,
                      float* final_state, float* ckpt_states, int ckpt_stride,
                      void* stream) {
    return prefill_pooled(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens,
                          H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, KDA_DECAY_CHANNEL,
                          nullptr, nullptr, nullptr, 0.f, stream);
}

int kda_chunk_prefill_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const float* log_alpha, const uint16_t* beta,
                         const float* init_state,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int num_seqs, int total_tokens, int H, int Dk, int Dv,
                         void* out, int out_dtype,
                         float* final_state, float* ckpt_states, int ckpt_stride,
                         int decay, const int32_t* start_pos, const int32_t* start_pos_host,
                         const float* out_norm_gamma, float out_norm_eps, void* stream) {
    return prefill_pooled(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens,
                          H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, decay, start_pos,
                          start_pos_host, out_norm_gamma, out_norm_eps, stream);
}

int kda_chunk_prefill_segmented_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const float* log_alpha, const uint16_t* beta,
                                   const float* init_state,
                                   const int32_t* cu_seqlens_host, int num_seqs, int total_tokens,
                                   int H, int Dk, int Dv,
                                   void* out, int out_dtype,
                                   float* final_state, float* ckpt_states, int ckpt_stride,
                                   int decay, const int32_t* start_pos_host, int segments,
                                   const float* out_norm_gamma, float out_norm_eps, void* stream) {
    if (segments < 1 || segments > KDA_MAX_SEGMENTS || num_seqs < 0 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs > KDA_MAX_SEGMENTED_SEQS) return KDA_ERR_UNSUPPORTED;
    // (the checks of the plain call; the host cu_seqlens stands in for the device copy, which
    // this entry point builds itself)
    int rc = check_prefill_args(q, k, v, log_alpha, beta, init_state, cu_seqlens_host, cu_seqlens_host, num_seqs,
                                total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, decay);
    if (rc != KDA_OK) return rc;
    if (Dk != Dv) return KDA_ERR_UNSUPPORTED;
    if (out_norm_gamma && (!aligned16(out_norm_gamma) || !(out_norm_eps >= 0.f) || !(out_norm_eps < 3.0e38f)))
        return KDA_ERR_INVALID_ARG;
    if (start_pos_host)
        for (int n = 0; n < num_seqs; ++n)
            if (start_pos_host[n] < 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;

    SegPlan plan;
    rc = plan_segments(cu_seqlens_host, start_pos_host, num_seqs, segments, ckpt_states ? ckpt_stride : 0, &plan);
    if (rc != KDA_OK) return rc;
    const int n_seg = plan.n_seg;
    const bool split = !plan.g0.empty();

    // device index arrays: segment bounds, start positions, roles, owning sequences; the
    // call's own cu_seqlens and start positions
    std::vector<int32_t> ucu(cu_seqlens_host, cu_seqlens_host + num_seqs + 1), usp(num_seqs, 0);
    if (start_pos_host) usp.assign(start_pos_host, start_pos_host + num_seqs);
    const size_t n_idx = (split ? plan.cu.size() + plan.sp.size() + plan.role.size() + plan.seq.size() : 0) +
                         ucu.size() + usp.size();
    if (n_idx > static_cast<size_t>(kda::kSegIdxMax)) return KDA_ERR_UNSUPPORTED;
    kda::SegIdxBuf ib;
    ib.n = 0;
    int o_cu = 0, o_sp = 0, o_role = 0, o_seq = 0, o_ucu = 0, o_usp = 0;
    auto put = [&](const std::vector<int32_t>& x, int* off) {
        *off = ib.n;
        for (int32_t e : x) ib.v[ib.n++] = e;
    };
    if (split) { put(plan.cu, &o_cu); put(plan.sp, &o_sp); put(plan.role, &o_role); put(plan.seq, &o_seq); }
    put(ucu, &o_ucu); put(usp, &o_usp);

    int* status = nullptr;
    rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(&pool);
    if (rc != KDA_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t slot = static_cast<size_t>(H) * Dk * Dv * sizeof(float);
    const size_t slot_f = slot / sizeof(float);

    if (!split) {   // no sequence is long enough to split: one plain prefill
        int32_t* idx = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&idx), up(sizeof(int32_t) * ib.n), pool, st) !=
            cudaSuccess)
            return KDA_ERR_CUDA;
        rc = kda::launch_segment_setup(ib, idx, 0, 0, 0, H, Dk, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                       st) == 0 ? KDA_OK : KDA_ERR_CUDA;
        if (rc == KDA_OK)
            rc = prefill_pooled(q, k, v, log_alpha, beta, init_state, idx + o_ucu, ucu.data(), num_seqs, total_tokens,
                                H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, decay,
                                idx + o_usp, usp.data(), out_norm_gamma, out_norm_eps, stream);
        const bool freed = cudaFreeAsync(idx, st) == cudaSuccess;
        return rc != KDA_OK ? rc : (freed ? KDA_OK : KDA_ERR_CUDA);
    }

    // scratch: index arrays | run A initial states | identities | Phi | S_start | run F final
    // states | checkpoints of runs A and F | zero v | bound partial sums | skip lists A, B, F
    const size_t o_idx = 0;
    const size_t o_zin = o_idx + up(sizeof(int32_t) * ib.n);
    const size_t o_idn = o_zin + slot * n_seg;
    const size_t o_phi = o_idn + slot * n_seg;
    const size_t o_sst = o_phi + slot * n_seg;
    const size_t o_fin = o_sst + slot * n_seg;
    const size_t o_ck = o_fin + slot * n_seg;
    const size_t o_zv = o_ck + slot * static_cast<size_t>(2 * plan.n_ck);
    const size_t o_part = o_zv + up(static_cast<size_t>(total_tokens) * H * Dv * 2);
    const size_t o_ska = o_part + up(sizeof(float) * static_cast<size_t>(n_seg) * H * kda::kSegBoundBlocks);
    const size_t o_skb = o_ska + up(sizeof(int) * static_cast<size_t>(n_seg) * H);
    const size_t o_skf = o_skb + up(sizeof(int) * static_cast<size_t>(n_seg) * H);
    const size_t total = o_skf + up(sizeof(int) * static_cast<size_t>(n_seg) * H);
    uint8_t* ws = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), total, pool, st) != cudaSuccess) return KDA_ERR_CUDA;
    int32_t* idx = reinterpret_cast<int32_t*>(ws + o_idx);
    float* zin = reinterpret_cast<float*>(ws + o_zin);
    float* idn = reinterpret_cast<float*>(ws + o_idn);
    float* phi = reinterpret_cast<float*>(ws + o_phi);
    float* sst = reinterpret_cast<float*>(ws + o_sst);
    float* fin = reinterpret_cast<float*>(ws + o_fin);
    float* ck = reinterpret_cast<float*>(ws + o_ck);
    uint16_t* zv = reinterpret_cast<uint16_t*>(ws + o_zv);
    float* part = reinterpret_cast<float*>(ws + o_part);
    int* skip_a = reinterpret_cast<int*>(ws + o_ska);
    int* skip_b = reinterpret_cast<int*>(ws + o_skb);
    int* skip_f = reinterpret_cast<int*>(ws + o_skf);
    auto finish = [&](int r) {
        const bool freed = cudaFreeAsync(ws, st) == cudaSuccess;
        return r != KDA_OK ? r : (freed ? KDA_OK : KDA_ERR_CUDA);
    };
    const int32_t* seg_cu = idx + o_cu;
    const int32_t* seg_sp = idx + o_sp;
    const bool want_ck = ckpt_states != nullptr && ckpt_stride > 0;

    if (kda::launch_segment_setup(ib, idx, n_seg, o_role, o_seq, H, Dk, init_state, idn, zin, sst, skip_a, skip_f,
                                  st) != 0)
        return finish(KDA_ERR_CUDA);
    // A: a split sequence's segments but its last; its first segment from the sequence's initial
    // state (outputs, norm and checkpoints final), the others from zeros (B); the end state of
    // segment g lands in S_start slot g + 1
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaStream_t side = nullptr;
    if (side_stream(&side) != KDA_OK || cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess || cudaEventRecord(fork, st) != cudaSuccess) {
        if (fork) cudaEventDestroy(fork);
        if (join) cudaEventDestroy(join);
        return finish(KDA_ERR_CUDA);
    }
    rc = prefill_pooled(q, k, v, log_alpha, beta, zin, seg_cu, plan.cu.data(), n_seg, total_tokens, H, Dk, Dv, out,
                        out_dtype, sst + slot_f, want_ck ? ck : nullptr, want_ck ? ckpt_stride : 0, decay, seg_sp,
                        plan.sp.data(), out_norm_gamma, out_norm_eps, stream, skip_a);
    // beside run A, on the SMs it leaves idle: v = 0 where run B may read it (the middle
    // segments), and which transitions cannot matter (their norm bound is below fp32
    // rounding: run B leaves them out and the chain takes the segment's B alone)
    bool side_ok = cudaStreamWaitEvent(side, fork, 0) == cudaSuccess;
    for (size_t z = 0; side_ok && z < plan.g0.size(); ++z) {
        const int g0 = plan.g0[z], P = plan.np[z];
        if (P < 3) continue;
        const size_t t0 = static_cast<size_t>(plan.cu[g0 + 1]), t1 = static_cast<size_t>(plan.cu[g0 + P - 1]);
        if (t1 > t0) side_ok = cudaMemsetAsync(zv + t0 * H * Dv, 0, (t1 - t0) * H * Dv * 2, side) == cudaSuccess;
    }
    side_ok = side_ok &&
              kda::launch_segment_bound(k, log_alpha, beta, decay, H, Dk, seg_cu, idx + o_role, n_seg, part, skip_b,
                                        side) == 0;
    side_ok = side_ok && cudaEventRecord(join, side) == cudaSuccess && cudaStreamWaitEvent(st, join, 0) == cudaSuccess;
    cudaEventDestroy(fork);
    cudaEventDestroy(join);
    if (!side_ok) {            // the scratch must outlive whatever reached the side stream
        cudaStreamSynchronize(side);
        return finish(rc != KDA_OK ? rc : KDA_ERR_CUDA);
    }
    if (rc != KDA_OK) return finish(rc);
    // B: the middle segments, from S_start = I with v = 0 (Phi), where the bound does not rule them out
    rc = prefill_pooled(q, k, zv, log_alpha, beta, idn, seg_cu, plan.cu.data(), n_seg, total_tokens, H, Dk, Dv, out,
                        out_dtype, phi, nullptr, 0, decay, seg_sp, plan.sp.data(), nullptr, 0.f, stream, skip_b);
    if (rc != KDA_OK) return finish(rc);
    // chain: S_start[p + 1] = Phi_p S_start[p] + B_p along every split sequence
    kda::SegChainBuf cb;
    cb.n = 0;
    for (size_t z = 0; z < plan.g0.size(); ++z)
        if (plan.np[z] >= 3) { cb.g0[cb.n] = plan.g0[z]; cb.np[cb.n] = plan.np[z]; ++cb.n; }
    if (cb.n > 0 && kda::launch_segment_chain(cb, phi, skip_b, sst, H, Dk, st) != 0) return finish(KDA_ERR_CUDA);
    // F: every segment but the first of a split sequence, from its S_start
    rc = prefill_pooled(q, k, v, log_alpha, beta, sst, seg_cu, plan.cu.data(), n_seg, total_tokens, H, Dk, Dv, out,
                        out_dtype, fin, want_ck ? ck + static_cast<size_t>(plan.n_ck) * slot_f : nullptr,
                        want_ck ? ckpt_stride : 0, decay, seg_sp, plan.sp.data(), out_norm_gamma, out_norm_eps, stream,
                        skip_f);
    if (rc != KDA_OK) return finish(rc);
    // each sequence's final state: its last segment's, from run F
    if (final_state)
        for (int n = 0; n < num_seqs; ++n)
            if (cudaMemcpyAsync(final_state + static_cast<size_t>(n) * slot_f,
                                fin + static_cast<size_t>(plan.last[n]) * slot_f, slot, cudaMemcpyDeviceToDevice,
                                st) != cudaSuccess)
                return finish(KDA_ERR_CUDA);
    // the call's checkpoints, in order: runs of consecutive kept slots, one copy each
    if (want_ck) {
        const std::vector<int>& keep = plan.keep;
        for (size_t i = 0, u = 0; i < keep.size();) {
            size_t j = i + 1;
            while (j < keep.size() && keep[j] == keep[j - 1] + 1) ++j;
            if (cudaMemcpyAsync(ckpt_states + u * slot_f, ck + static_cast<size_t>(keep[i]) * slot_f, (j - i) * slot,
                                cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return finish(KDA_ERR_CUDA);
            u += j - i;
            i = j;
        }
    }
    return finish(KDA_OK);
}

int kda_chunk_prefill_segmented(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const float* log_alpha, const uint16_t* beta,
                                const float* init_state,
                                int total_tokens, int H, int Dk, int Dv,
                                void* out, int out_dtype,
                                float* final_state, float* ckpt_states, int ckpt_stride,
                                int decay, int start_pos, int segments,
                                const float* out_norm_gamma, float out_norm_eps, void* stream) {
    if (total_tokens < 0 || start_pos < 0) return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(start_pos) + total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    const int32_t cu1[2] = {0, total_tokens};
    const int32_t sp1[1] = {start_pos};
    return kda_chunk_prefill_segmented_ex(q, k, v, log_alpha, beta, init_state, cu1, 1, total_tokens, H, Dk, Dv, out,
                                          out_dtype, final_state, ckpt_states, ckpt_stride, decay, sp1, segments,
                                          out_norm_gamma, out_norm_eps, stream);
}

int kda_chunk_prefill_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              const float* log_alpha, const uint16_t* beta,
                              const float* init_state,
                              const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                              int num_seqs, int total_tokens, int H, int Dk, int Dv,
                              void* out, int out_dtype,
                              float* final_state, float* ckpt_states, int ckpt_stride,
                              void* stream) {
    int rc = check_prefill_args(q, k, v, log_alpha, beta, init_state, cu_seqlens, cu_seqlens_host, num_seqs,
                                total_tokens, H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride,
                                KDA_DECAY_CHANNEL);
    if (rc != KDA_OK || num_seqs == 0) return rc;
    if (static_cast<int64_t>(num_seqs) * H > KDA_NOALLOC_MAX_SEQ_HEADS) return KDA_ERR_UNSUPPORTED;
    int* status = nullptr;
    uint8_t* scratch = nullptr;
    rc = device_setup(&status, &scratch);
    if (rc != KDA_OK) return rc;
    rc = kda::launch_prefill(q, k, v, log_alpha, beta, init_state, cu_seqlens, num_seqs, total_tokens, H, Dk, Dv,
                             out, out_dtype == KDA_OUT_F32, final_state, ckpt_states, ckpt_stride,
                             KDA_DECAY_CHANNEL, nullptr, nullptr, 0.f, scratch, nullptr, 0, status,
                             static_cast<cudaStream_t>(stream));
    return rc == 0 ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_step(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const float* log_alpha, const uint16_t* beta,
                    float* state, void* out, int out_dtype,
                    int N, int H, int Dk, int Dv, void* stream) {
    if (N < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (out_dtype != KDA_OUT_BF16 && out_dtype != KDA_OUT_F32) return KDA_ERR_INVALID_ARG;
    if (!head_dims_ok(Dk, Dv)) return KDA_ERR_UNSUPPORTED;
    if (Dk != Dv) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, log_alpha, beta, state, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * H >= (int64_t(1) << 31)) return KDA_ERR_INVALID_ARG;
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    rc = kda::launch_decode(q, k, v, log_alpha, beta, state, out, out_dtype == KDA_OUT_F32, N, H, Dk,
                            static_cast<cudaStream_t>(stream));
    return rc == 0 ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_multi(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const float* log_alpha, const uint16_t* beta,
                     float* state_pool, int num_slots, const int32_t* state_slots,
                     const int32_t* num_tokens, int commit,
                     void* out, int out_dtype,
                     int N, int K, int H, int Dk, int Dv, int decay, void* stream) {
    if (N < 0 || K < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (decay != KDA_DECAY_CHANNEL && decay != KDA_DECAY_HEAD && decay != KDA_DECAY_NONE) return KDA_ERR_INVALID_ARG;
    if (out_dtype != KDA_OUT_BF16 && out_dtype != KDA_OUT_F32) return KDA_ERR_INVALID_ARG;
    if (commit != 0 && commit != 1) return KDA_ERR_INVALID_ARG;
    if (!head_dims_ok(Dk, Dv)) return KDA_ERR_UNSUPPORTED;
    if (Dk != Dv) return KDA_ERR_UNSUPPORTED;
    if (N == 0 || K == 0) return KDA_OK;
    if (!q || !k || !v || !beta || !state_pool || !out) return KDA_ERR_INVALID_ARG;
    if ((decay == KDA_DECAY_NONE) != (log_alpha == nullptr)) return KDA_ERR_INVALID_ARG;
    if (!state_slots && num_slots < N) return KDA_ERR_INVALID_ARG;
    if (num_slots == 0) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, log_alpha, beta, state_pool, out};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if ((state_slots && (reinterpret_cast<uintptr_t>(state_slots) & 3u)) ||
        (num_tokens && (reinterpret_cast<uintptr_t>(num_tokens) & 3u)))
        return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(N) * K * H >= (int64_t(1) << 31) || static_cast<int64_t>(N) * H >= (int64_t(1) << 31))
        return KDA_ERR_INVALID_ARG;
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    rc = kda::launch_decode_multi(q, k, v, log_alpha, beta, state_pool, num_slots, state_slots, num_tokens, commit,
                                  out, out_dtype == KDA_OUT_F32, N, K, H, Dk, decay, status,
                                  static_cast<cudaStream_t>(stream));
    return rc == 0 ? KDA_OK : KDA_ERR_CUDA;
}

int kda_prepare_inputs(const uint16_t* xq, const uint16_t* xk, const uint16_t* xv,
                       const float* conv_w, const uint16_t* conv_state,
                       const float* a_raw, const uint16_t* b_raw,
                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                       int num_seqs, int total_tokens, int H, int D, int conv_act,
                       uint16_t* q, uint16_t* k, uint16_t* v, float* log_alpha, uint16_t* beta,
                       void* stream) {
    if (num_seqs < 0 || total_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return KDA_ERR_UNSUPPORTED;
    if (conv_act != 0 && conv_act != 1) return KDA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!cu_seqlens || !cu_seqlens_host)) return KDA_ERR_INVALID_ARG;
    if (num_seqs > 0) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
        for (int n = 0; n < num_seqs; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
    } else if (total_tokens != 0) {
        return KDA_ERR_INVALID_ARG;
    }
    if (total_tokens == 0) return KDA_OK;
    const void* need[] = {xq, xk, xv, conv_w, a_raw, b_raw, q, k, v, log_alpha, beta};
    for (const void* p : need)
        if (!p) return KDA_ERR_INVALID_ARG;
    const void* a16[] = {xq, xk, xv, conv_w, conv_state, a_raw, q, k, v, log_alpha};
    for (const void* p : a16)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(b_raw) & 1u) || (reinterpret_cast<uintptr_t>(beta) & 1u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(total_tokens) * H * D >= (int64_t(1) << 40)) return KDA_ERR_INVALID_ARG;
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    rc = kda::launch_prepare_inputs(xq, xk, xv, conv_w, conv_state, a_raw, b_raw, cu_seqlens, num_seqs, total_tokens,
                                    H, D, conv_act, q, k, v, log_alpha, beta, status,
                                    static_cast<cudaStream_t>(stream));
    return rc == 0 ? KDA_OK : KDA_ERR_CUDA;
}

int kda_output_norm(const void* o, int o_dtype, const float* gamma, float eps,
                    uint16_t* y, int total_tokens, int H, int Dv, void* stream) {
    if (total_tokens < 0 || H <= 0 || !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
    if (o_dtype != KDA_OUT_BF16 && o_dtype != KDA_OUT_F32) return KDA_ERR_INVALID_ARG;
    if (Dv != 64 && Dv != 128) return KDA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return KDA_OK;
    if (!o || !gamma || !y) return KDA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(gamma) || !aligned16(y)) return KDA_ERR_INVALID_ARG;
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    rc = kda::launch_output_norm(o, o_dtype == KDA_OUT_F32, gamma, eps, y, total_tokens, H, Dv,
                                 static_cast<cudaStream_t>(stream));
    return rc == 0 ? KDA_OK : KDA_ERR_CUDA;
}

int kda_debug_expire_wait(unsigned long long limit_ns, void* stream) {
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    if (limit_ns < 1000000ull) limit_ns = 1000000ull;
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_device_status(void* stream) {
    int* status = nullptr;
    int rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_kda_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_kda_status, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return value;
}

}  // extern "C"
