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
int launch_segment_setup(const SegIdxBuf& ib, int32_t* idx, float* ident, int n_ident, float* zinit, int n_zinit,
                         const float* init_state, int* flags, int n_flags, int n_flags_set, int H, int D,
                         cudaStream_t stream);
int launch_segment_chain(const float* phi, const int* skip, float* sst, int P, int H, int D, cudaStream_t stream);
int launch_segment_bound(const uint16_t* k, const float* la, const uint16_t* beta, int decay, int H, int D,
                         const int32_t* seg_start, int nseg, int lead, float* partial, int* skip,
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

// The plan of a segmented prefill.
//   b[0..P]   segment bounds, tokens from the prompt's start, on the absolute 64-token chunk
//             grid (equal chunk counts, the last segment shorter; P = 1 when fewer than 3
//             segments result, which runs one plain prefill)
//   b1a       segment 1's start rounded down to a multiple of 8 tokens; the runs that start
//             there (B and F) put a short leading sequence [b1a, b1) first (lead = 1) so that
//             every per-token row they address stays 16-byte aligned; it is skipped
//   checkpoints: run A (segments 0 .. P-2) writes n_ck_a slots and run F (the leading
//             sequence, then segments 1 .. P-1) n_ck_f; keep[i] is the slot, in run A's slots
//             followed by run F's, of the prompt's i-th own checkpoint (segment 0's come from
//             run A, the rest from run F; every run also writes one slot at each of its
//             sequences' ends, which is kept only at a stride multiple or the prompt's end)
struct SegPlan {
    int P = 1;
    std::vector<int32_t> b;
    int32_t b1a = 0;
    int lead = 0;
    std::vector<int> keep;
    int64_t n_ck_a = 0, n_ck_f = 0;
};

int plan_segments(int total_tokens, int start_pos, int segments, int ckpt_stride, SegPlan* out) {
    if (segments < 1 || segments > KDA_MAX_SEGMENTS || start_pos < 0 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_stride < 0 || ckpt_stride % 64 != 0) return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(start_pos) + total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    const int C = 64;
    const int64_t s0 = start_pos, T = total_tokens;
    const int64_t c_first = s0 / C, c_end = (s0 + T + C - 1) / C;
    const int64_t n_chunks = T > 0 ? c_end - c_first : 0;
    int P = 1;
    int64_t per = n_chunks;
    if (segments >= 3 && n_chunks >= 3) {
        per = (n_chunks + segments - 1) / segments;
        P = static_cast<int>((n_chunks + per - 1) / per);
        if (P < 3) P = 1;
    }
    std::vector<int32_t> b(P + 1);
    for (int p = 0; p <= P; ++p) {
        const int64_t x = C * (c_first + p * per) - s0;
        b[p] = static_cast<int32_t>(x < 0 ? 0 : (x > T ? T : x));
    }
    b[0] = 0;
    b[P] = total_tokens;
    const int32_t b1a = P >= 3 ? (b[1] & ~7) : 0;
    const int lead = (P >= 3 && b1a < b[1]) ? 1 : 0;
    std::vector<int> keep;
    int64_t n_a = 0, n_f = 0;
    if (ckpt_stride > 0 && P >= 3) {
        // slots of one sequence [a, e) (absolute positions): the stride multiples strictly inside,
        // then its end; `own` marks those that are the prompt's checkpoints
        auto slots = [&](int64_t a, int64_t e, bool last, int64_t base, int64_t* n, bool own_any) {
            for (int64_t m = (a / ckpt_stride + 1) * ckpt_stride; m < e; m += ckpt_stride) {
                if (own_any) keep.push_back(static_cast<int>(base + *n));
                ++*n;
            }
            if (own_any && (e % ckpt_stride == 0 || last)) keep.push_back(static_cast<int>(base + *n));
            ++*n;
        };
        for (int p = 0; p <= P - 2; ++p) slots(s0 + b[p], s0 + b[p + 1], false, 0, &n_a, p == 0);
        if (lead) slots(s0 + b1a, s0 + b[1], false, 0, &n_f, false);
        for (int p = 1; p <= P - 1; ++p) slots(s0 + b[p], s0 + b[p + 1], p == P - 1, n_a, &n_f, true);
        const int32_t cu1[2] = {0, total_tokens};
        const int32_t sp1[1] = {start_pos};
        if (static_cast<int64_t>(keep.size()) != kda_ckpt_count_ex(cu1, sp1, 1, ckpt_stride)) return KDA_ERR_INVALID_ARG;
    }
    out->P = P;
    out->b = std::move(b);
    out->b1a = b1a;
    out->lead = lead;
    out->keep = std::move(keep);
    out->n_ck_a = n_a;
    out->n_ck_f = n_f;
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
    if (!bounds) return KDA_ERR_INVALID_ARG;
    SegPlan plan;
    const int rc = plan_segments(total_tokens, start_pos, segments, ckpt_stride, &plan);
    if (rc != KDA_OK) return rc;
    if (ckpt_slots && static_cast<int64_t>(plan.keep.size()) > ckpt_slots_cap) return KDA_ERR_INVALID_ARG;
    for (int p = 0; p <= plan.P; ++p) bounds[p] = plan.b[p];
    if (ckpt_slots)
        for (size_t i = 0; i < plan.keep.size(); ++i) ckpt_slots[i] = plan.keep[i];
    return plan.P;
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

int kda_chunk_prefill_segmented(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const float* log_alpha, const uint16_t* beta,
                                const float* init_state,
                                int total_tokens, int H, int Dk, int Dv,
                                void* out, int out_dtype,
                                float* final_state, float* ckpt_states, int ckpt_stride,
                                int decay, int start_pos, int segments,
                                const float* out_norm_gamma, float out_norm_eps, void* stream) {
    if (segments < 1 || segments > KDA_MAX_SEGMENTS || start_pos < 0 || total_tokens < 0) return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(start_pos) + total_tokens > INT32_MAX) return KDA_ERR_INVALID_ARG;
    const int32_t cu1[2] = {0, total_tokens};
    // (the one-sequence checks of the plain call; cu1 stands in for the device cu_seqlens,
    // which this entry point builds itself)
    int rc = check_prefill_args(q, k, v, log_alpha, beta, init_state, cu1, cu1, 1, total_tokens, H, Dk, Dv, out,
                                out_dtype, final_state, ckpt_states, ckpt_stride, decay);
    if (rc != KDA_OK) return rc;
    if (Dk != Dv) return KDA_ERR_UNSUPPORTED;
    if (out_norm_gamma && (!aligned16(out_norm_gamma) || !(out_norm_eps >= 0.f) || !(out_norm_eps < 3.0e38f)))
        return KDA_ERR_INVALID_ARG;

    SegPlan plan;
    rc = plan_segments(total_tokens, start_pos, segments, ckpt_states ? ckpt_stride : 0, &plan);
    if (rc != KDA_OK) return rc;
    const int P = plan.P;
    const std::vector<int32_t>& b = plan.b;

    const int32_t b1a = plan.b1a;
    const int lead = plan.lead;
    const int nA = P >= 3 ? P - 1 : 0;              // run A: segments 0 .. P-2
    const int nB = P >= 3 ? P - 2 + lead : 0;       // run B: [leading,] segments 1 .. P-2
    const int nF = P >= 3 ? P - 1 + lead : 0;       // run F: [leading,] segments 1 .. P-1

    // host index arrays (cu_seqlens, start positions) of the runs; B and F count tokens from b1a
    std::vector<int32_t> a_cu, a_sp, b_cu, b_sp, f_cu, f_sp, bnd(b.begin(), b.end()), sp0{start_pos};
    if (P >= 3) {
        for (int p = 0; p <= nA; ++p) a_cu.push_back(b[p]);
        for (int p = 0; p < nA; ++p) a_sp.push_back(start_pos + b[p]);
        b_cu.push_back(0);
        f_cu.push_back(0);
        if (lead) {
            b_cu.push_back(b[1] - b1a); b_sp.push_back(start_pos + b1a);
            f_cu.push_back(b[1] - b1a); f_sp.push_back(start_pos + b1a);
        }
        for (int p = 1; p <= P - 2; ++p) { b_cu.push_back(b[p + 1] - b1a); b_sp.push_back(start_pos + b[p]); }
        for (int p = 1; p <= P - 1; ++p) { f_cu.push_back(b[p + 1] - b1a); f_sp.push_back(start_pos + b[p]); }
    }
    if (a_cu.size() + a_sp.size() + b_cu.size() + b_sp.size() + f_cu.size() + f_sp.size() + bnd.size() + sp0.size() >
        static_cast<size_t>(kda::kSegIdxMax))
        return KDA_ERR_INVALID_ARG;
    kda::SegIdxBuf ib;
    ib.n = 0;
    int o_acu = 0, o_asp = 0, o_bcu = 0, o_bsp = 0, o_fcu = 0, o_fsp = 0, o_bnd = 0, o_sp0 = 0;
    auto put = [&](const std::vector<int32_t>& x, int* off) {
        *off = ib.n;
        for (int32_t e : x) ib.v[ib.n++] = e;
    };
    put(a_cu, &o_acu); put(a_sp, &o_asp); put(b_cu, &o_bcu); put(b_sp, &o_bsp); put(f_cu, &o_fcu); put(f_sp, &o_fsp);
    put(bnd, &o_bnd); put(sp0, &o_sp0);

    const std::vector<int>& keep = plan.keep;
    const int64_t n_ck = plan.n_ck_a + plan.n_ck_f;

    int* status = nullptr;
    rc = device_setup(&status);
    if (rc != KDA_OK) return rc;
    cudaMemPool_t pool = nullptr;
    rc = workspace_pool(&pool);
    if (rc != KDA_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);

    // scratch: index arrays | run A initial states | run B identities | Phi | S_start |
    // run F final states | checkpoints of runs A and F | zero v of run B | bound partial sums |
    // run B skip list | run F skip list
    const size_t slot = static_cast<size_t>(H) * Dk * Dv * sizeof(float);
    const size_t slot_f = slot / sizeof(float);
    const bool zinit_needed = P >= 3 && init_state != nullptr;
    const int64_t tB = P >= 3 ? static_cast<int64_t>(b[P - 1]) - b1a : 0;
    const int64_t tF = P >= 3 ? static_cast<int64_t>(total_tokens) - b1a : 0;
    const int nseg = P >= 3 ? P - 2 : 0;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t o_idx = 0;
    const size_t o_zin = o_idx + up(sizeof(int32_t) * ib.n);
    const size_t o_idn = o_zin + (zinit_needed ? slot * nA : 0);
    const size_t o_phi = o_idn + slot * nB;
    const size_t o_sst = o_phi + slot * nB;
    const size_t o_fin = o_sst + (P >= 3 ? slot * P : 0);
    const size_t o_ck = o_fin + slot * nF;
    const size_t o_zv = o_ck + slot * static_cast<size_t>(n_ck);
    const size_t o_part = o_zv + up(static_cast<size_t>(tB) * H * Dv * 2);
    const size_t o_skip = o_part + up(sizeof(float) * static_cast<size_t>(nseg) * H * kda::kSegBoundBlocks);
    const size_t o_fskip = o_skip + up(sizeof(int) * static_cast<size_t>(nB) * H);
    const size_t total = o_fskip + up(sizeof(int) * static_cast<size_t>(nF) * H);
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
    int* skip = reinterpret_cast<int*>(ws + o_skip);
    int* fskip = reinterpret_cast<int*>(ws + o_fskip);

    auto finish = [&](int r) {
        const bool freed = cudaFreeAsync(ws, st) == cudaSuccess;
        return r != KDA_OK ? r : (freed ? KDA_OK : KDA_ERR_CUDA);
    };
    if (kda::launch_segment_setup(ib, idx, idn, nB, zin, zinit_needed ? nA : 0, init_state, fskip, nF * H, lead * H,
                                  H, Dk, st) != 0)
        return finish(KDA_ERR_CUDA);
    if (P < 3)   // one plain prefill
        return finish(prefill_pooled(q, k, v, log_alpha, beta, init_state, idx + o_bnd, bnd.data(), 1, total_tokens,
                                     H, Dk, Dv, out, out_dtype, final_state, ckpt_states, ckpt_stride, decay,
                                     idx + o_sp0, sp0.data(), out_norm_gamma, out_norm_eps, stream));

    if (tB > 0 && cudaMemsetAsync(zv, 0, static_cast<size_t>(tB) * H * Dv * 2, st) != cudaSuccess)
        return finish(KDA_ERR_CUDA);
    // which transitions cannot matter (their norm bound is below fp32 rounding): those runs are
    // skipped and their segment starts from B alone
    if (kda::launch_segment_bound(k, log_alpha, beta, decay, H, Dk, idx + o_bnd + 1, nseg, lead, part, skip, st) != 0)
        return finish(KDA_ERR_CUDA);
    const size_t la_row = decay == KDA_DECAY_CHANNEL ? static_cast<size_t>(Dk) : 1;
    const size_t osz = out_dtype == KDA_OUT_F32 ? 4 : 2;
    const size_t tok = static_cast<size_t>(b1a) * H;        // token rows before b1a
    // A: segments 0 .. P-2.  Segment 0 starts from the prompt's initial state, so its outputs
    // (normed, if asked) and checkpoints are final; its final state lands in S_start[1], and
    // B_p (p >= 1, from zeros) in S_start[p + 1]
    rc = prefill_pooled(q, k, v, log_alpha, beta, zinit_needed ? zin : nullptr, idx + o_acu, a_cu.data(), nA,
                        b[P - 1], H, Dk, Dv, out, out_dtype, sst + slot_f, ckpt_states ? ck : nullptr,
                        ckpt_states ? ckpt_stride : 0, decay, idx + o_asp, a_sp.data(), out_norm_gamma, out_norm_eps,
                        stream);
    if (rc != KDA_OK) return finish(rc);
    // B: from S_start = I with v = 0, tokens from b1a on (the leading sequence, if any, first)
    rc = prefill_pooled(q + tok * Dk, k + tok * Dk, zv, log_alpha ? log_alpha + tok * la_row : nullptr, beta + tok,
                        idn, idx + o_bcu, b_cu.data(), nB, static_cast<int>(tB), H, Dk, Dv,
                        static_cast<uint8_t*>(out) + tok * Dv * osz, out_dtype, phi, nullptr, 0, decay,
                        idx + o_bsp, b_sp.data(), nullptr, 0.f, stream, skip);
    if (rc != KDA_OK) return finish(rc);
    // chain: S_start[p + 1] = Phi_p S_start[p] + B_p, p = 1 .. P-2 (Phi_p in slot p - 1 + lead)
    if (kda::launch_segment_chain(phi + static_cast<size_t>(lead) * slot_f, skip + lead * H, sst, P, H, Dk, st) != 0)
        return finish(KDA_ERR_CUDA);
    // F: segments 1 .. P-1 from S_start[1 ..] (the leading sequence, skipped, takes slot 0)
    rc = prefill_pooled(q + tok * Dk, k + tok * Dk, v + tok * Dv, log_alpha ? log_alpha + tok * la_row : nullptr,
                        beta + tok, sst + (lead ? 0 : slot_f), idx + o_fcu, f_cu.data(), nF, static_cast<int>(tF), H,
                        Dk, Dv, static_cast<uint8_t*>(out) + tok * Dv * osz, out_dtype, fin,
                        ckpt_states ? ck + static_cast<size_t>(plan.n_ck_a) * slot_f : nullptr,
                        ckpt_states ? ckpt_stride : 0, decay, idx + o_fsp, f_sp.data(), out_norm_gamma, out_norm_eps,
                        stream, lead ? fskip : nullptr);
    if (rc != KDA_OK) return finish(rc);
    if (final_state &&
        cudaMemcpyAsync(final_state, fin + static_cast<size_t>(nF - 1) * slot_f, slot, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
        return finish(KDA_ERR_CUDA);
    // the prompt's checkpoints, in order: runs of consecutive kept slots, one copy each
    for (size_t i = 0, u = 0; i < keep.size();) {
        size_t j = i + 1;
        while (j < keep.size() && keep[j] == keep[j - 1] + 1) ++j;
        if (cudaMemcpyAsync(ckpt_states + u * (slot / sizeof(float)), ck + static_cast<size_t>(keep[i]) * (slot / sizeof(float)),
                            (j - i) * slot, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return finish(KDA_ERR_CUDA);
        u += j - i;
        i = j;
    }
    return finish(KDA_OK);
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
