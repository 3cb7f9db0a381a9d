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
// (cudaGetSymbolAddress) and caches it; that first call should therefore be
// made before any stream capture begins.
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
void* g_scratch_addr[kMaxDevices];

// device address of g_scratch on the current device (cached per device)
int scratch_address(int device, void** out)
{
    if (device < 0 || device >= kMaxDevices) return GATO_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GATO_ERR_CUDA;
        }
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return GATO_OK;
}

size_t round64(size_t x)
{
    const size_t r = (x + 63) / 64 * 64;
    return r ? r : 64;
}

// The same workspace layout gato_create uses, placed at `base` (or, with
// base == nullptr, only sized).  Returns the bytes needed.
size_t carve(Work& w, int M, int N, int n, int m, float* base)
{
    w.M = M; w.N = N; w.n = n; w.m = m;
    const size_t K = (size_t)(N - 1);
    w.sNnn = round64((size_t)N * n * n);
    w.sKnn = round64(K * n * n);
    w.sKmm = round64(K * m * m);
    w.sKnm = round64(K * n * m);
    w.sNn = round64((size_t)N * n);
    w.sN = round64((size_t)N);
    w.sKm = round64(K * m);
    w.sK2 = (size_t)N * (GATO_MAX_ALPHA + 1);
    float** fields[] = {&w.Qinv, &w.Rinv, &w.O, &w.V, &w.D, &w.L, &w.Linv, &w.Pd, &w.Po, &w.Nh,
                        &w.dlow,
                        &w.rhs[0].gamma, &w.rhs[0].ghat, &w.rhs[0].avec, &w.rhs[0].bvec,
                        &w.rhs[1].gamma, &w.rhs[1].ghat, &w.rhs[1].avec, &w.rhs[1].bvec,
                        &w.q2, &w.r2, &w.e2, &w.s02, &w.dlam, &w.ddX, &w.ddU};
    const size_t strides[] = {w.sNnn, w.sKmm, w.sKnn, w.sKnm, w.sNnn, w.sNnn, w.sNnn,
                              w.sNnn, w.sKnn, w.sKnn, w.sN, w.sNn, w.sNn, w.sNn, w.sKm,
                              w.sNn, w.sNn, w.sNn, w.sKm,
                              w.sNn, w.sKm, w.sNn, w.sNn, w.sNn, w.sNn, w.sKm};
    const int nf = (int)(sizeof(strides) / sizeof(strides[0]));
    size_t total = 0;
    for (int i = 0; i < nf; ++i) {
        if (base) *fields[i] = base + total;
        total += strides[i] * (size_t)M;
    }
    if (base) w.mpart = (float2*)(base + total);
    total += 2 * w.sK2 * (size_t)M;
    if (base) w.queue = (int*)(base + total);
    total += 64;  // work counters
    return total * sizeof(float);
}

bool params_ok(const gato_params* p)
{
    if (!p) return false;
    if (!(p->pcg_eps >= 0.f) || p->pcg_max_iters < 0) return false;
    if (p->stop_rule < GATO_STOP_RESIDUAL || p->stop_rule > GATO_STOP_SCALED) return false;
    if (p->refine_steps < 0 || p->refine_steps > 16) return false;
    if (p->n_alpha < 1 || p->n_alpha > GATO_MAX_ALPHA) return false;
    if (!(p->beta > 1.f) || !(p->mu >= 0.f)) return false;
    if (p->merit_threads < 32 || p->merit_threads > 256 || p->merit_threads % 32) return false;
    if (!(p->refine_eps >= 0.f)) return false;
    if (p->merit_kernel != GATO_MERIT_FUSED && p->merit_kernel != GATO_MERIT_PER_CANDIDATE)
        return false;
    return true;
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
    if (!params_ok(p) || !Q || !q || !s0 || !dX || !lambda || !iters || !merit || !best ||
        !status)
        return GATO_ERR_INVALID_ARG;
    if (N > 1 && (!R || !r || !A || !B || !e || !dU)) return GATO_ERR_INVALID_ARG;
    Work probe;
    if (carve(probe, M, N, n, m, nullptr) > (size_t)GATO_NOALLOC_MAX_BYTES)
        return GATO_ERR_UNSUPPORTED;

    gato_handle h{};  // on the stack: nothing is allocated
    if (cudaGetDevice(&h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               h.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, h.device) !=
            cudaSuccess)
        return GATO_ERR_CUDA;
    void* base = nullptr;
    const int rc = scratch_address(h.device, &base);
    if (rc != GATO_OK) return rc;
    h.base = base;
    h.bytes = carve(h.w, M, N, n, m, (float*)base);

    cudaStream_t st = (cudaStream_t)stream;
    Work& w = h.w;
    cudaError_t err = gato::launch_form_matrices(&h, Q, R, A, B, status, st);
    if (err == cudaSuccess) err = gato::launch_form_rhs(&h, 0, q, r, e, s0, (size_t)n, st);
    if (err == cudaSuccess)
        err = gato::launch_pcg_ex(&h, p, 0, nullptr, lambda, dX, dU, iters, 0, status, st);
    gato_params pc = *p;
    if (p->refine_eps > 0.f) pc.pcg_eps = p->refine_eps;
    for (int k = 0; k < p->refine_steps && err == cudaSuccess; ++k) {
        err = gato::launch_kkt_residual(&h, Q, R, q, r, A, B, e, s0, dX, dU, lambda, st);
        if (err == cudaSuccess)
            err = gato::launch_form_rhs(&h, 1, w.q2, w.r2, w.e2, w.s02, (size_t)n, st);
        if (err == cudaSuccess)
            err = gato::launch_pcg_ex(&h, &pc, 1, nullptr, w.dlam, w.ddX, w.ddU, iters, 1,
                                      status, st);
        if (err == cudaSuccess) err = gato::launch_accumulate(&h, lambda, dX, dU, iters, st);
    }
    if (err == cudaSuccess)
        err = gato::launch_merit(&h, p, Q, R, q, r, A, B, e, s0, dX, dU, merit, best, status, st);
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GATO_OK : GATO_ERR_CUDA;
}
