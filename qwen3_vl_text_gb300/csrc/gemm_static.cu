// Projection GEMM for callers that cannot allocate device memory.
//
// h3enc_op_gemm needs a caller-allocated workspace for the stream-K split of its
// last partial wave.  Some callers have no way to provide one: code that runs inside
// another framework's allocator callback or after a memory pool has reserved the
// whole device, plugins that are handed only input and output buffers, and hosts
// that forbid cudaMalloc after start-up.  h3enc_op_gemm_noalloc runs the same
// kernel with the same schedule but takes its scratch from a fixed array that
// lives in this library's device image: every GPU that loads the library holds
// it (kScratchBytes) until the process exits.
#include <cstdio>
#include <mutex>

#include "../../include/h3enc_ops.h"
#include "kernels.h"

namespace {

// Partials of the stream-K phase: two 128 x 256 fp32 slots per SM, then one flag per SM, then
// the launch epoch and the finished-CTA counter (found right after the flags of the SMs in use).
constexpr int kMaxSlots = 160;                                      // SMs the array is sized for
constexpr size_t kSlotBytes = 128 * 256 * sizeof(float);            // 128 KiB
constexpr size_t kFlagOffset = (size_t)2 * kMaxSlots * kSlotBytes + 256;
constexpr size_t kFlagWords = kMaxSlots + 2;
constexpr size_t kScratchBytes = kFlagOffset + kFlagWords * sizeof(uint32_t);  // 40 MiB + 904 B

static __device__ __align__(256) unsigned char g_gemm_scratch[kScratchBytes];

using h3::kMaxDevices;
std::mutex g_setup_mutex;
unsigned char *g_scratch_addr[kMaxDevices] = {nullptr};

thread_local char g_error[256];

// Device address of the scratch array on the current device.  The first call on
// a device looks the address up (the host-side name is only a stand-in) and
// zero-fills the flags with a memset ordered on the caller's stream (no device-wide
// synchronisation); it refuses to run while that stream is being captured.  Later
// calls return the cached address.
h3enc_status scratch_for_current_device(cudaStream_t stream, unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: no CUDA device: %s", cudaGetErrorString(e));
        return H3ENC_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: device index %d above %d", dev, kMaxDevices - 1);
        return H3ENC_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &cs);
        if (e != cudaSuccess) {
            snprintf(g_error, sizeof g_error, "gemm_noalloc: cannot query the stream: %s", cudaGetErrorString(e));
            return H3ENC_ERR_CUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) {
            snprintf(g_error, sizeof g_error,
                     "gemm_noalloc: the first call on device %d sets up the scratch array and cannot run "
                     "inside a stream capture; make one call on this device before capturing", dev);
            return H3ENC_ERR_UNSUPPORTED;
        }
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_gemm_scratch);
        if (e != cudaSuccess || !p) {
            snprintf(g_error, sizeof g_error, "gemm_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return H3ENC_ERR_CUDA;
        }
        // a flag equal to the epoch of a launch means "partial written": flags, epoch and counter
        // start from zero
        e = cudaMemsetAsync(static_cast<unsigned char *>(p) + kFlagOffset, 0, kFlagWords * sizeof(uint32_t), stream);
        if (e != cudaSuccess) {
            snprintf(g_error, sizeof g_error, "gemm_noalloc: clearing the flags failed: %s", cudaGetErrorString(e));
            return H3ENC_ERR_CUDA;
        }
        g_scratch_addr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_scratch_addr[dev];
    return H3ENC_OK;
}

}  // namespace

extern "C" {

H3ENC_API int64_t h3enc_op_gemm_noalloc_scratch_bytes(void) { return (int64_t)kScratchBytes; }

H3ENC_API const char *h3enc_op_gemm_noalloc_last_error(void) { return g_error; }

H3ENC_API h3enc_status h3enc_op_gemm_noalloc(const void *A, const void *W, void *C, int32_t M, int32_t N, int32_t K,
                                             int32_t epilogue, const void *R, const void *DS,
                                             const int32_t *vis_rank, int32_t n_vis, int32_t *status,
                                             void *stream) {
    g_error[0] = 0;
    if (M < 0 || N <= 0 || K <= 0 || N % 256 || K % 8 || epilogue < 0 || epilogue > 3) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: bad sizes or epilogue");
        return H3ENC_ERR_INVALID_ARG;
    }
    if (M == 0) return H3ENC_OK;
    if (!A || !W || !C || ((epilogue == H3ENC_EPI_RESIDUAL || epilogue == H3ENC_EPI_RESIDUAL_DS) && !R) ||
        (epilogue == H3ENC_EPI_RESIDUAL_DS && DS && !vis_rank)) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: NULL operand");
        return H3ENC_ERR_INVALID_ARG;
    }
    const int sms = h3::device_num_sms();
    if (sms <= 0) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: cannot query the SM count");
        return H3ENC_ERR_CUDA;
    }
    // the split needs two 128 KiB slots and one flag per SM: a device with more SMs than the array
    // is sized for needs more scratch than the array holds and is refused
    if (sms > kMaxSlots) {
        snprintf(g_error, sizeof g_error,
                 "gemm_noalloc: this device has %d SMs and needs %zu scratch bytes; the static scratch holds %zu "
                 "(%d SMs) - use h3enc_op_gemm with a workspace",
                 sms, h3::gemm_workspace_bytes(sms), kScratchBytes, kMaxSlots);
        return H3ENC_ERR_UNSUPPORTED;
    }
    unsigned char *scratch = nullptr;
    h3enc_status s = scratch_for_current_device(static_cast<cudaStream_t>(stream), &scratch);
    if (s != H3ENC_OK) return s;
    CUtensorMap ta, tw;
    if (!h3::make_tmap_rows(&ta, A, M, K, h3::gemm_box_rows_a()) ||
        !h3::make_tmap_rows(&tw, W, N, K, h3::gemm_box_rows_w())) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: operands not 16-byte aligned or the driver refused the map");
        return H3ENC_ERR_INVALID_ARG;
    }
    h3::GemmPlan p{};
    p.tmA = &ta;
    p.tmW = &tw;
    p.M = M;
    p.N = N;
    p.K = K;
    p.epi = epilogue;
    p.C = static_cast<h3::bf16 *>(C);
    p.ldc = epilogue == H3ENC_EPI_SWIGLU ? N / 2 : N;
    p.R = static_cast<const h3::bf16 *>(R);
    p.DS = static_cast<const h3::bf16 *>(DS);
    p.vis_rank = vis_rank;
    p.n_vis = n_vis;
    p.status = status;
    p.num_sms = sms;
    // slots from the start of the array, flags at the fixed offset the set-up cleared (both indexed by CTA)
    p.part = reinterpret_cast<float *>(scratch);
    p.flags = reinterpret_cast<uint32_t *>(scratch + kFlagOffset);
    cudaError_t e = h3::launch_gemm(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        snprintf(g_error, sizeof g_error, "gemm_noalloc: launch failed: %s", cudaGetErrorString(e));
        return H3ENC_ERR_CUDA;
    }
    return H3ENC_OK;
}

}  // extern "C"
