/*
 * kda_debug.h -- test hook for the library's failure detection.
 *
 * Every device-side wait in the KDA kernels is bounded: when a wait expires the
 * kernel records KDA_ERR_TIMEOUT in the device status word and returns early,
 * so the CUDA context stays usable and kda_device_status() reports the
 * failure.  This entry point exercises exactly that path on demand, without
 * faulting, trapping or hanging the GPU.
 */
#ifndef KDA_DEBUG_H_
#define KDA_DEBUG_H_

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kda_debug_expire_wait -- launch one small kernel on `stream` (a cudaStream_t
 * as void*) whose thread waits on an mbarrier phase that nothing completes.
 * The wait gives up after limit_ns nanoseconds (clamped to 1 ms .. 1 s), the
 * kernel records KDA_ERR_TIMEOUT and returns.  Returns KDA_OK when the launch
 * was enqueued (the timeout is then visible through kda_device_status()),
 * KDA_ERR_UNSUPPORTED on a device without sm_103a, KDA_ERR_CUDA on a launch
 * failure.  The paper describes no counterpart; this exists for testing.
 */
int kda_debug_expire_wait(unsigned long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_DEBUG_H_ */
