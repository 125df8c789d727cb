// Library-wide plumbing: last-error text, the per-device status word, wait
// timeouts, device checks, tensor-map encoding, and the failure-detection
// self test (a bounded wait on a barrier phase that never completes).
#include <cstdlib>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "vae_common.cuh"

namespace vae {

namespace {
thread_local char g_last_error[1024] = {0};
std::mutex g_mu;
constexpr int kMaxDevices = 64;
DevStatus* g_status_ptr[kMaxDevices] = {nullptr};
int g_sm_count[kMaxDevices] = {0};
int g_dev_ok[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 unsupported
unsigned long long g_timeout_ns = 4000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct CtxFns {
    CtxGetCurrentFn current = nullptr;
    CtxGetIdFn id = nullptr;
    CtxFns() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            id = reinterpret_cast<CtxGetIdFn>(f);
    }
};
CtxOnce g_status_once;
}  // namespace

unsigned long long context_id() {
    static const CtxFns fns;  // resolved once (thread-safe static initialisation)
    if (fns.current == nullptr || fns.id == nullptr) return 0;
    CUcontext c = nullptr;
    if (fns.current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    if (fns.id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The status word every kernel of this library writes on a timed-out wait.
__device__ DevStatus g_dev_status[1];

int set_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_last_error[0] = 0; }

static int current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return set_error(VAE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (*dev < 0 || *dev >= kMaxDevices) return set_error(VAE_ERR_UNSUPPORTED, "device index %d", *dev);
    return VAE_OK;
}

DevStatus* device_status_ptr() {
    int dev;
    if (current_device(&dev) != VAE_OK) return nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (g_status_ptr[dev] == nullptr || !g_status_once.done(dev)) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_dev_status);
        if (e != cudaSuccess) {
            set_error(VAE_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<DevStatus*>(p);
        g_status_once.mark(dev);
    }
    return g_status_ptr[dev];
}

unsigned long long wait_timeout_ns() { return g_timeout_ns; }

bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VAE_PDL");
        return e != nullptr && e[0] == '1';
    }();
    return on;
}

int sm_count() {
    int dev;
    if (current_device(&dev) != VAE_OK) return 0;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int check_device() {
    int dev;
    int rc = current_device(&dev);
    if (rc != VAE_OK) return rc;
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e1 != cudaSuccess || e2 != cudaSuccess)
            return set_error(VAE_ERR_CUDA, "cudaDeviceGetAttribute: %s",
                             cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_dev_ok[dev] < 0)
            return set_error(VAE_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                             dev, major, minor);
    }
    if (g_dev_ok[dev] < 0) return set_error(VAE_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
    return VAE_OK;
}

int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* gaddr,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                             cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return set_error(VAE_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
    }
    cuuint64_t gd[5];
    cuuint64_t gs[4];
    cuuint32_t bx[5];
    cuuint32_t es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(gaddr), gd, gs,
                          bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(VAE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d), rank %d", static_cast<int>(r),
                         rank);
    return VAE_OK;
}

// One thread waits, bounded, on the first phase of a barrier that expects
// one arrival nobody makes. The wait runs out and records the timeout.
__global__ void selftest_wait_kernel(DevStatus* st, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns, st, kWhereSelftest);
    }
}

}  // namespace vae

using namespace vae;

extern "C" {

const char* vae_version(void) { return "vae-igemm-gb300 0.1 (sm_103a)"; }

const char* vae_last_error(void) { return g_last_error; }

int vae_set_wait_timeout_ns(unsigned long long ns) {
    g_timeout_ns = ns == 0 ? 4000000000ull : ns;
    return VAE_OK;
}

int vae_sync_status(vae_stream_t stream) {
    clear_error();
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    DevStatus* p = device_status_ptr();
    if (p == nullptr) return VAE_ERR_CUDA;
    VAE_CUDA_CHECK(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    DevStatus h{};
    VAE_CUDA_CHECK(cudaMemcpy(&h, p, sizeof(h), cudaMemcpyDeviceToHost));
    if (h.code != 0) {
        DevStatus z{};
        VAE_CUDA_CHECK(cudaMemcpy(p, &z, sizeof(z), cudaMemcpyHostToDevice));
        return set_error(VAE_ERR_DEVICE_TIMEOUT,
                         "a bounded device wait ran out (site %d, block %d, parity %d)", h.where, h.info0,
                         h.info1);
    }
    return VAE_OK;
}

int vae_selftest_wait_timeout(unsigned long long timeout_ns, vae_stream_t stream) {
    clear_error();
    int rc = check_device();
    if (rc != VAE_OK) return rc;
    if (timeout_ns == 0 || timeout_ns > 10000000000ull)
        return set_error(VAE_ERR_ARG, "timeout_ns must be in (0, 1e10]");
    DevStatus* p = device_status_ptr();
    if (p == nullptr) return VAE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    selftest_wait_kernel<<<1, 32, 0, s>>>(p, timeout_ns);
    VAE_CUDA_CHECK(cudaGetLastError());
    return vae_sync_status(stream);
}

}  // extern "C"
