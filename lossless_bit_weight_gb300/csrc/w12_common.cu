// Host-side plumbing shared by every W12 entry point: status names, device check, shape and
// tensor validation.
#include <cudaTypedefs.h>

#include <mutex>

#include "w12_internal.cuh"

namespace w12 {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_device_ok[kMaxDevices];  // 0 unknown, 1 ok, -1 wrong architecture
std::mutex g_mu;
}  // namespace

w12_status require_device(int *sm_count) {
    int dev = 0;
    W12_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return W12_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        W12_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
        W12_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
        W12_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_sm_count[dev] = sms;
    }
    if (g_device_ok[dev] != 1) return W12_ERR_DEVICE;
    if (sm_count) *sm_count = g_sm_count[dev];
    return W12_OK;
}

// The driver's tensor-map encoder, looked up once through the runtime (no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

w12_status check_shape(int N, int K) {
    if (N < 1 || K < 1) return W12_ERR_INVALID_ARG;
    if (K % 8 != 0) return W12_ERR_UNSUPPORTED_SHAPE;
    // escape-list offsets are 32-bit: keep the weight count (and so every offset) below 2^31
    if (static_cast<int64_t>(N) * K > (int64_t(1) << 31)) return W12_ERR_UNSUPPORTED_SHAPE;
    return W12_OK;
}

w12_status check_tensor(const w12_tensor *t) {
    if (!t) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(t->N, t->K));
    if (t->n_tiles != ceil_div(t->N, kTileN) || t->k_tiles != ceil_div(t->K, kTileK))
        return W12_ERR_INVALID_ARG;
    if (!t->records || !t->base_exp || !t->rec_esc_off || !t->esc_off) return W12_ERR_INVALID_ARG;
    if (t->n_esc < 0 || t->n_rec_esc < 0) return W12_ERR_INVALID_ARG;
    if (t->n_rec_esc > 0 && !t->rec_esc) return W12_ERR_INVALID_ARG;
    if (t->n_esc > 0 && (!t->esc_k || !t->esc_bits)) return W12_ERR_INVALID_ARG;
    if (!aligned16(t->records)) return W12_ERR_INVALID_ARG;
    if (t->rec_esc && !aligned16(t->rec_esc)) return W12_ERR_INVALID_ARG;
    return W12_OK;
}

}  // namespace w12

extern "C" const char *w12_status_str(w12_status s) {
    switch (s) {
        case W12_OK: return "W12_OK";
        case W12_ERR_INVALID_ARG: return "W12_ERR_INVALID_ARG";
        case W12_ERR_UNSUPPORTED_SHAPE: return "W12_ERR_UNSUPPORTED_SHAPE";
        case W12_ERR_WORKSPACE: return "W12_ERR_WORKSPACE";
        case W12_ERR_CUDA: return "W12_ERR_CUDA";
        case W12_ERR_MISMATCH: return "W12_ERR_MISMATCH";
        case W12_ERR_TIMEOUT: return "W12_ERR_TIMEOUT";
        case W12_ERR_DEVICE: return "W12_ERR_DEVICE";
    }
    return "W12_ERR_UNKNOWN";
}

extern "C" w12_status w12_tensor_shape(int N, int K, w12_tensor *t, size_t *records_bytes,
                                       size_t *base_exp_bytes) {
    using namespace w12;
    if (!t) return W12_ERR_INVALID_ARG;
    W12_TRY(check_shape(N, K));
    t->N = N;
    t->K = K;
    t->n_tiles = static_cast<int32_t>(ceil_div(N, kTileN));
    t->k_tiles = static_cast<int32_t>(ceil_div(K, kTileK));
    if (records_bytes)
        *records_bytes = static_cast<size_t>(t->n_tiles) * t->k_tiles * kRecordBytes;
    if (base_exp_bytes) *base_exp_bytes = static_cast<size_t>(t->n_tiles) * kTileN;
    return W12_OK;
}
