// gato_noalloc.cu -- gato_solve_kkt_noalloc: the whole batched KKT solve with
// no device allocation at call time.
//
// Some callers cannot allocate device memory while they run: a real-time MPC
// loop whose memory is fixed when it starts (an allocation in the control
// loop costs unbounded time), or a host framework that owns every device
// allocation and hands libraries only the buffers it made.  For them the
// solver's scratch (the Schur blocks, preconditioner factors, right-hand
// sides, refinement buffers and merit partial sums that gato_create would
// allocate) lives in one file-scope device array of GATO_NOALLOC_MAX_BYTES,
// reserved on every GPU that loads the library until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in symbol, not a device address.  The first call on each device,
// with that device current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and caches it together with the identifier of the
// CUDA context it belongs to; that first call should therefore be made
// before any stream capture begins.  A device reset (cudaDeviceReset)
// destroys that context and the module is loaded again, possibly elsewhere,
// in the next one: a later call sees a different context identifier and
// looks the address up again instead of passing a stale pointer.
//
// All calls share the one array and it keeps whatever the last call left in
// it.  The solve writes every scratch entry before reading it, so nothing
// needs clearing between calls; but calls whose work overlaps on the GPU
// (different streams, or different host threads) race on the array and
// must be serialised by the caller.
#include <mutex>

#include "gato_internal.cuh"

using gato::Work;

namespace {

static __device__ __align__(256) unsigned char g_scratch[GATO_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct Cached {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    void* addr;
};
Cached g_cache[kMaxDevices];

// the driver's current-context queries, reached through the runtime so that
// the library needs no link against the driver library
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// identifier of the current context, 0 when there is none or it cannot be read
unsigned long long current_context_id()
{
    if (!g_ctx_get_current || !g_ctx_get_id) {
        cudaDriverEntryPointQueryResult q1, q2;
        void* f1 = nullptr;
        void* f2 = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2) {
            cudaGetLastError();
            return 0;
        }
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != 0 || !ctx || g_ctx_get_id(ctx, &id) != 0) return 0;
    return id;
}

// device address of g_scratch on the current device: cached per device and
// looked up again when the device's context has changed since
int scratch_address(int device, void** out)
{
    if (device < 0 || device >= kMaxDevices) return GATO_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    Cached& c = g_cache[device];
    if (c.addr && c.ctx_id != 0 && current_context_id() == c.ctx_id) {
        *out = c.addr;
        return GATO_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return GATO_ERR_CUDA;
    }
    c.addr = p;
    c.ctx_id = current_context_id();  // the lookup made the context current
    *out = p;
    return GATO_OK;
}

}  // namespace

extern "C" int gato_solve_kkt_noalloc(const gato_params* p, int M, int N, int n, int m,
                                      const float* Q, const float* R, const float* q,
                                      const float* r, const float* A, const float* B,
                                      const float* e, const float* s0, float* dX, float* dU,
                                      float* lambda, int32_t* iters, float* merit,
                                      int32_t* best, uint32_t* status, void* stream)
{
    if (M < 1 || N < 1 || n < 1 || m < 1) return GATO_ERR_INVALID_ARG;
    if (n > GATO_MAX_STATE || m > GATO_MAX_CONTROL) return GATO_ERR_UNSUPPORTED;
    if (!gato::params_valid(p) || !Q || !q || !s0 || !dX || !lambda || !iters || !merit ||
        !best || !status)
        return GATO_ERR_INVALID_ARG;
    if (N > 1 && (!R || !r || !A || !B || !e || !dU)) return GATO_ERR_INVALID_ARG;
    Work probe;
    if (gato::carve_workspace(probe, M, N, n, m, nullptr) > (size_t)GATO_NOALLOC_MAX_BYTES)
        return GATO_ERR_UNSUPPORTED;

    gato_handle h{};  // on the stack: nothing is allocated, no timing events
    if (cudaGetDevice(&h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device) !=
            cudaSuccess)
        return GATO_ERR_CUDA;
    if (!gato::sizes_supported(probe, p, h.smem_optin)) return GATO_ERR_UNSUPPORTED;
    void* base = nullptr;
    const int rc = scratch_address(h.device, &base);
    if (rc != GATO_OK) return rc;
    h.base = base;
    h.bytes = gato::carve_workspace(h.w, M, N, n, m, (float*)base);

    const cudaError_t err = gato::run_solve_kkt(&h, p, Q, R, q, r, A, B, e, s0, dX, dU, lambda,
                                                iters, merit, best, status, (cudaStream_t)stream);
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GATO_OK : GATO_ERR_CUDA;
}
