// gato_api.cu -- the extern "C" entry points declared in include/gato.h:
// argument checks, the workspace allocation, stage ordering on the caller's
// stream and the optional per-stage CUDA-event timing.
#include <stdlib.h>
#include <string.h>

#include "gato_internal.cuh"

using gato::Work;

namespace gato {

namespace {
size_t round64(size_t x)
{
    const size_t r = (x + 63) / 64 * 64;
    return r ? r : 64;
}
}  // namespace

size_t carve_workspace(Work& w, int M, int N, int n, int m, float* base)
{
    w.M = M; w.N = N; w.n = n; w.m = m;
    w.status = nullptr;
    const size_t K = (size_t)(N - 1);
    w.sNnn = round64((size_t)N * n * n);
    w.sKnn = round64(K * n * n);
    w.sKmm = round64(K * m * m);
    w.sKnm = round64(K * n * m);
    w.sNn = round64((size_t)N * n);
    w.sN = round64((size_t)N);
    w.sKm = round64(K * m);
    w.sK2 = (size_t)N * (GATO_MAX_ALPHA + 1);  // float2 units
    float* ints = nullptr;  // three int arrays of M (SQP best, iterations, counter)
    // one allocation: (per-solve floats of each array) x M, in this order
    float** fields[] = {&w.Qinv, &w.Rinv, &w.O, &w.V, &w.D, &w.L, &w.Linv, &w.Pd, &w.Po, &w.Nh,
                        &w.dlow,
                        &w.rhs[0].gamma, &w.rhs[0].ghat, &w.rhs[0].avec, &w.rhs[0].bvec,
                        &w.rhs[1].gamma, &w.rhs[1].ghat, &w.rhs[1].avec, &w.rhs[1].bvec,
                        &w.q2, &w.r2, &w.e2, &w.s02, &w.dlam, &w.ddX, &w.ddU,
                        &w.Bd, &w.Be, &w.By, &w.Bv, &w.Bg,
                        &w.Qd, &w.qt, &w.rt, &w.et, &w.s0t, &w.Jk, &w.sdX, &w.sdU,
                        &w.smerit, &ints};
    const size_t strides[] = {w.sNnn, w.sKmm, w.sKnn, w.sKnm, w.sNnn, w.sNnn, w.sNnn,
                              w.sNnn, w.sKnn, w.sKnn, w.sN, w.sNn, w.sNn, w.sNn, w.sKm,
                              w.sNn, w.sNn, w.sNn, w.sKm,
                              w.sNn, w.sKm, w.sNn, w.sNn, w.sNn, w.sNn, w.sKm,
                              w.sNnn, w.sNnn, w.sNnn, w.sNn, w.sNn,
                              w.sNnn, w.sNn, w.sKm, w.sNn, w.sNn, w.sN, w.sNn, w.sKm,
                              32, 4};
    static_assert(sizeof(fields) / sizeof(fields[0]) == sizeof(strides) / sizeof(strides[0]),
                  "one stride per workspace array");
    const int nf = (int)(sizeof(strides) / sizeof(strides[0]));
    size_t total = 0;
    for (int i = 0; i < nf; ++i) {
        if (base) *fields[i] = base + total;
        total += strides[i] * (size_t)M;
    }
    if (base) {
        w.sbest = reinterpret_cast<int*>(ints);
        w.siters = w.sbest + M;
        w.sqpt = w.sbest + 2 * M;
    }
    if (base) w.mpart = (float2*)(base + total);
    total += 2 * w.sK2 * (size_t)M;  // merit partials
    if (base) w.queue = (int*)(base + total);
    total += 64;                     // work counters
    if (base) w.mcount = (int*)(base + total);
    total += (size_t)M;              // merit: blocks arrived per solve
    return total * sizeof(float);
}

bool params_valid(const gato_params* p)
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
    if (p->linsys < GATO_LINSYS_AUTO || p->linsys > GATO_LINSYS_BDSV_CHRONO) return false;
    if (p->bdsv_horizon < 1) return false;
    if (p->pcg_precision != GATO_PCG_PRECISION_FP32 && p->pcg_precision != GATO_PCG_PRECISION_FF)
        return false;
    if (p->refine_solver != GATO_REFINE_SOLVER_SAME &&
        p->refine_solver != GATO_REFINE_SOLVER_DIRECT)
        return false;
    return true;
}

bool sizes_supported(const Work& w, const gato_params* p, int smem_limit)
{
    if (p->pcg_precision != GATO_PCG_PRECISION_FF) return true;
    if (linsys_for(p, w.N) != GATO_LINSYS_PCG) return true;
    return pcg_ff_fits(w.N, w.n, (size_t)smem_limit);
}

int linsys_for(const gato_params* p, int N)
{
    if (p->linsys == GATO_LINSYS_AUTO)
        return N >= p->bdsv_horizon ? GATO_LINSYS_BDSV : GATO_LINSYS_PCG;
    return p->linsys;
}

namespace {
void record(gato_handle* h, int i, cudaStream_t st)
{
    if (!h->timing) return;
    cudaEventRecord(h->ev[i], st);
    h->ev_used[i] = 1;
}
}  // namespace

cudaError_t run_kkt_core(gato_handle* h, const gato_params* p, const float* Q_form,
                         const float* Q_merit, const float* R, const float* q, const float* r,
                         const float* A, const float* B, const float* e, const float* s0,
                         const float* lambda0, float* dX, float* dU, float* lambda,
                         int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                         cudaStream_t st, bool timed)
{
    Work& w = h->w;
    w.status = status;
    h->pcg_ran = h->refine_ran = 0;
    const int ls = linsys_for(p, w.N);
    const bool direct = ls != GATO_LINSYS_PCG;
    // corrections by substitution with the direct solve's factors: those of the
    // main solve, or (GATO_REFINE_SOLVER_DIRECT after a PCG solve) the
    // cyclic-reduction factorisation of the same S, formed once.  That
    // factorisation needs only the formation's blocks, so with a side stream
    // it is forked off once the main PCG is launched and runs on the SMs the
    // PCG leaves idle (its stream has the lowest priority); the corrections
    // join it before their first substitution
    const bool direct_ref =
        direct || (p->refine_solver == GATO_REFINE_SOLVER_DIRECT && p->refine_steps > 0);
    const int ls_ref = direct ? ls : GATO_LINSYS_BDSV;
    const bool fork_factor = direct_ref && !direct && h->side;
    bool joined = false;
    cudaError_t err = launch_form_matrices(h, Q_form, R, A, B, status, st);
    if (err == cudaSuccess) err = launch_form_rhs(h, 0, q, r, e, s0, (size_t)w.n, st);
    if (timed) record(h, 1, st);
    if (err == cudaSuccess) {
        if (direct) {
            err = launch_bdsv_factor(h, ls, status, st);
            if (err == cudaSuccess)
                err = launch_bdsv_solve(h, ls, 0, lambda, dX, dU, iters, 0, status, st);
        } else {
            if (fork_factor) err = cudaEventRecord(h->ev_fork, st);
            if (err == cudaSuccess)
                err = launch_pcg_ex(h, p, 0, lambda0, lambda, dX, dU, iters, 0, status, st);
            if (err == cudaSuccess && fork_factor) {
                err = cudaStreamWaitEvent(h->side, h->ev_fork, 0);
                if (err == cudaSuccess) err = launch_bdsv_factor(h, ls_ref, status, h->side);
                if (err == cudaSuccess) err = cudaEventRecord(h->ev_join, h->side);
            }
        }
    }
    if (timed) record(h, 2, st);
    // PCG corrections are solved to refine_eps on the preconditioned residual
    // (r^T Phi^-1 r): a correction only needs a digit, and that test costs no
    // residual-norm evaluation
    gato_params pc = *p;
    if (p->refine_eps > 0.f) pc.pcg_eps = p->refine_eps;
    pc.stop_rule = GATO_STOP_PRECOND;
    pc.pcg_precision = GATO_PCG_PRECISION_FP32;
    if (err == cudaSuccess && direct_ref && !direct && !fork_factor)
        err = launch_bdsv_factor(h, ls_ref, status, st);
    for (int k = 0; k < p->refine_steps && err == cudaSuccess; ++k) {
        err = launch_kkt_residual(h, Q_form, R, q, r, A, B, e, s0, dX, dU, lambda, st);
        if (err == cudaSuccess)
            err = launch_form_rhs(h, 1, w.q2, w.r2, w.e2, w.s02, (size_t)w.n, st);
        if (err == cudaSuccess && fork_factor && k == 0) {
            err = cudaStreamWaitEvent(st, h->ev_join, 0);
            joined = err == cudaSuccess;
        }
        if (err == cudaSuccess) {
            if (direct_ref)
                err = launch_bdsv_solve(h, ls_ref, 1, w.dlam, w.ddX, w.ddU, iters, 1, status,
                                        st);
            else
                err = launch_pcg_ex(h, &pc, 1, nullptr, w.dlam, w.ddX, w.ddU, iters, 1, status,
                                    st);
        }
        if (err == cudaSuccess) err = launch_accumulate(h, lambda, dX, dU, iters, st);
    }
    // after an error the caller's stream still waits for the side stream, so
    // that nothing of this call runs on after it (the event completes at once
    // when nothing was recorded)
    if (fork_factor && !joined) cudaStreamWaitEvent(st, h->ev_join, 0);
    if (timed && p->refine_steps > 0) record(h, 3, st);
    if (err == cudaSuccess)
        err = launch_merit(h, p, Q_merit, R, q, r, A, B, e, s0, dX, dU, merit, best, status, st);
    if (timed) record(h, 4, st);
    return err;
}

cudaError_t run_solve_kkt(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                          const float* q, const float* r, const float* A, const float* B,
                          const float* e, const float* s0, float* dX, float* dU, float* lambda,
                          int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                          cudaStream_t st)
{
    return run_kkt_core(h, p, Q, Q, R, q, r, A, B, e, s0, nullptr, dX, dU, lambda, iters, merit,
                        best, status, st, true);
}

}  // namespace gato

namespace {

using gato::params_valid;

int cuda_fail(cudaError_t e) { return e == cudaSuccess ? GATO_OK : GATO_ERR_CUDA; }

// the [N-1] arrays may be NULL only when N == 1
bool lq_ok(const gato_handle* h, const float* Q, const float* R, const float* q,
           const float* r, const float* A, const float* B, const float* e, const float* s0)
{
    if (!Q || !q || !s0) return false;
    if (h->w.N > 1 && (!R || !r || !A || !B || !e)) return false;
    return true;
}

void record(gato_handle* h, int i, cudaStream_t st)
{
    if (!h->timing) return;
    cudaEventRecord(h->ev[i], st);
    h->ev_used[i] = 1;
}

void begin_timing(gato_handle* h, cudaStream_t st)
{
    h->pcg_ran = h->refine_ran = 0;
    if (!h->timing) return;
    for (int i = 0; i < 5; ++i) h->ev_used[i] = 0;
    record(h, 0, st);
}

int unsupported_or_fail(cudaError_t e)
{
    if (e == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return cuda_fail(e);
}

bool sqp_params_valid(const gato_sqp_params* sp)
{
    if (!sp || sp->iters < 1) return false;
    if (!(sp->rho_factor > 1.f) || !(sp->rho_min >= 0.f) || !(sp->rho_max >= sp->rho_min))
        return false;
    return true;
}

struct SqpArgs {
    const float *Q, *R, *q, *r, *A, *B, *c, *xs;
    float *X, *U, *lambda, *rho, *merit_hist;
    int32_t* iters_hist;
    uint32_t* status;
};

// one SQP iteration: expansion, the damped KKT solve, line search, step
cudaError_t sqp_iteration(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                          const SqpArgs& a, cudaStream_t st)
{
    Work& w = h->w;
    w.status = a.status;
    cudaError_t err = gato::launch_sqp_linearize(h, a.Q, a.R, a.q, a.r, a.A, a.B, a.c, a.xs,
                                                 a.X, a.U, a.rho, st);
    if (err == cudaSuccess)
        err = gato::run_kkt_core(h, p, w.Qd, a.Q, a.R, w.qt, w.rt, a.A, a.B, w.et, w.s0t,
                                 sp->warm_start ? a.lambda : nullptr, w.sdX, w.sdU, a.lambda,
                                 w.siters, w.smerit, w.sbest, a.status, st, false);
    if (err == cudaSuccess)
        err = gato::launch_sqp_step(h, p, sp, a.X, a.U, a.rho, a.merit_hist, a.iters_hist, st);
    return err;
}

// everything a recorded iteration depends on (parameters, pointers and the
// handle's kernel selections), in a zero-padded byte string
void sqp_key(unsigned char* key, const gato_handle* h, const gato_params* p,
             const gato_sqp_params* sp, const SqpArgs& a)
{
    static_assert(sizeof(gato_params) + sizeof(gato_sqp_params) + sizeof(SqpArgs) +
                          3 * sizeof(int) <= 512,
                  "key size");
    memset(key, 0, 512);
    const int kinds[3] = {h->pcg_kernel, h->bdsv_kernel, h->force_smem_form};
    gato_params pk;
    gato_sqp_params sk;
    memset(&pk, 0, sizeof(pk));
    memset(&sk, 0, sizeof(sk));
    pk = *p;
    sk = *sp;
    memcpy(key, &pk, sizeof(pk));
    memcpy(key + sizeof(pk), &sk, sizeof(sk));
    memcpy(key + sizeof(pk) + sizeof(sk), &a, sizeof(a));
    memcpy(key + sizeof(pk) + sizeof(sk) + sizeof(a), kinds, sizeof(kinds));
}

// records one iteration on the handle's private stream (nothing runs while
// recording) and instantiates it
cudaError_t record_sqp_graph(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                             const SqpArgs& a)
{
    if (h->sqp_exec) {
        cudaGraphExecDestroy(h->sqp_exec);
        h->sqp_exec = nullptr;
    }
    cudaError_t err = cudaSuccess;
    if (!h->capture_stream)
        err = cudaStreamCreateWithFlags(&h->capture_stream, cudaStreamNonBlocking);
    if (err != cudaSuccess) return err;
    err = cudaStreamBeginCapture(h->capture_stream, cudaStreamCaptureModeThreadLocal);
    if (err != cudaSuccess) return err;
    err = sqp_iteration(h, p, sp, a, h->capture_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t end = cudaStreamEndCapture(h->capture_stream, &g);
    if (err == cudaSuccess) err = end;
    if (err == cudaSuccess) err = cudaGraphInstantiate(&h->sqp_exec, g, 0);
    if (g) cudaGraphDestroy(g);
    if (err != cudaSuccess) {
        h->sqp_exec = nullptr;
        cudaGetLastError();
    }
    return err;
}

}  // namespace

extern "C" {

void gato_default_params(gato_params* p)
{
    if (!p) return;
    p->pcg_eps = 1e-6f;
    p->pcg_max_iters = 200;
    p->stop_rule = GATO_STOP_RESIDUAL;
    p->refine_steps = 0;
    p->n_alpha = 8;
    p->beta = 2.f;
    p->mu = 10.f;
    p->merit_threads = 64;
    p->refine_eps = 0.1f;
    p->merit_kernel = GATO_MERIT_FUSED;
    p->linsys = GATO_LINSYS_AUTO;
    p->bdsv_horizon = 256;
    p->pcg_precision = GATO_PCG_PRECISION_FP32;
    p->refine_solver = GATO_REFINE_SOLVER_SAME;
}

void gato_default_sqp_params(gato_sqp_params* sp)
{
    if (!sp) return;
    sp->iters = 10;
    sp->rho_factor = 10.f;
    sp->rho_min = 1e-8f;
    sp->rho_max = 10.f;
    sp->warm_start = 1;
    sp->use_graph = 1;
}

int gato_create(gato_handle** out, int M, int N, int n, int m)
{
    if (!out) return GATO_ERR_INVALID_ARG;
    *out = nullptr;
    if (M < 1 || N < 1 || n < 1 || m < 1) return GATO_ERR_INVALID_ARG;
    if (n > GATO_MAX_STATE || m > GATO_MAX_CONTROL) return GATO_ERR_UNSUPPORTED;
    gato_handle* h = (gato_handle*)calloc(1, sizeof(gato_handle));
    if (!h) return GATO_ERR_NO_MEMORY;
    if (cudaGetDevice(&h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               h->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) !=
            cudaSuccess) {
        free(h);
        return GATO_ERR_CUDA;
    }
    // room for the handle's workspace and for any partition of the batch into
    // parts, which are views into the same allocation
    h->bytes = gato::carve_workspace(h->w, M, N, n, m, nullptr) + gato::parts_extra_bytes();
    if (cudaMalloc(&h->base, h->bytes) != cudaSuccess) {
        cudaGetLastError();
        free(h);
        return GATO_ERR_NO_MEMORY;
    }
    gato::carve_workspace(h->w, M, N, n, m, (float*)h->base);
    for (int i = 0; i < 5; ++i) {
        if (cudaEventCreate(&h->ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(h->ev[j]);
            cudaFree(h->base);
            free(h);
            return GATO_ERR_CUDA;
        }
    }
    h->last.form_us = h->last.pcg_us = h->last.refine_us = h->last.merit_us = h->last.total_us =
        -1.f;
    int prc = gato::side_stream_create(&h->side, &h->ev_fork, &h->ev_join) == cudaSuccess
                  ? GATO_OK
                  : GATO_ERR_CUDA;
    if (prc == GATO_OK) prc = gato::parts_init(h);
    if (prc != GATO_OK) {
        if (h->side) cudaStreamDestroy(h->side);
        if (h->ev_fork) cudaEventDestroy(h->ev_fork);
        if (h->ev_join) cudaEventDestroy(h->ev_join);
        for (int i = 0; i < 5; ++i) cudaEventDestroy(h->ev[i]);
        cudaFree(h->base);
        free(h);
        return prc;
    }
    *out = h;
    return GATO_OK;
}

void gato_destroy(gato_handle* h)
{
    if (!h) return;
    gato::parts_free(h);
    if (h->sqp_exec) cudaGraphExecDestroy(h->sqp_exec);
    if (h->capture_stream) cudaStreamDestroy(h->capture_stream);
    if (h->side) cudaStreamDestroy(h->side);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    for (int i = 0; i < 5; ++i) cudaEventDestroy(h->ev[i]);
    cudaFree(h->base);
    free(h);
}

int gato_set_timing(gato_handle* h, int on)
{
    if (!h) return GATO_ERR_INVALID_ARG;
    h->timing = on ? 1 : 0;
    return GATO_OK;
}

int gato_set_pcg_kernel(gato_handle* h, int kind)
{
    if (!h || kind < GATO_PCG_AUTO || kind > GATO_PCG_QUAD) return GATO_ERR_INVALID_ARG;
    h->pcg_kernel = kind;
    return GATO_OK;
}

int gato_set_bdsv_kernel(gato_handle* h, int kind)
{
    if (!h || (kind != GATO_BDSV_KERNEL_AUTO && kind != GATO_BDSV_KERNEL_SHARED))
        return GATO_ERR_INVALID_ARG;
    h->bdsv_kernel = kind;
    return GATO_OK;
}

int gato_set_form_kernel(gato_handle* h, int kind)
{
    if (!h || (kind != GATO_FORM_AUTO && kind != GATO_FORM_SHARED)) return GATO_ERR_INVALID_ARG;
    h->force_smem_form = kind == GATO_FORM_SHARED;
    return GATO_OK;
}

int gato_get_stats(gato_handle* h, gato_stats* out)
{
    if (!h || !out) return GATO_ERR_INVALID_ARG;
    gato_stats s;
    s.form_us = s.pcg_us = s.refine_us = s.merit_us = s.total_us = -1.f;
    s.pcg_kernel = h->pcg_ran;
    s.refine_kernel = h->refine_ran;
    if (h->timing && h->ev_used[0]) {
        int last = 0;
        for (int i = 4; i > 0; --i)
            if (h->ev_used[i]) { last = i; break; }
        if (cudaEventSynchronize(h->ev[last]) != cudaSuccess) return GATO_ERR_CUDA;
        float ms;
        // stage i runs between the previous recorded event and event i
        int prev = 0;
        float* dst[5] = {nullptr, &s.form_us, &s.pcg_us, &s.refine_us, &s.merit_us};
        for (int i = 1; i < 5; ++i) {
            if (!h->ev_used[i]) continue;
            if (dst[i] && cudaEventElapsedTime(&ms, h->ev[prev], h->ev[i]) == cudaSuccess)
                *dst[i] = 1000.f * ms;
            prev = i;
        }
        if (cudaEventElapsedTime(&ms, h->ev[0], h->ev[last]) == cudaSuccess)
            s.total_us = 1000.f * ms;
    }
    h->last = s;
    *out = s;
    return GATO_OK;
}

int gato_form_schur(gato_handle* h, const float* Q, const float* R, const float* q,
                    const float* r, const float* A, const float* B, const float* e,
                    const float* s0, uint32_t* status, void* stream)
{
    if (!h || !status || !lq_ok(h, Q, R, q, r, A, B, e, s0)) return GATO_ERR_INVALID_ARG;
    h->w.status = status;
    cudaStream_t st = (cudaStream_t)stream;
    begin_timing(h, st);
    cudaError_t err = gato::launch_form_matrices(h, Q, R, A, B, status, st);
    if (err == cudaSuccess) err = gato::launch_form_rhs(h, 0, q, r, e, s0, (size_t)h->w.n, st);
    record(h, 1, st);
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return cuda_fail(err);
}

int gato_get_schur(gato_handle* h, float* S_diag, float* S_off, float* gamma,
                   float* Phi_diag, float* Phi_off, void* stream)
{
    if (!h) return GATO_ERR_INVALID_ARG;
    h->w.status = nullptr;
    const Work& w = h->w;
    cudaStream_t st = (cudaStream_t)stream;
    if ((Phi_diag || Phi_off) && h->phi_pending) {
        if (gato::launch_form_phi(h, st) != cudaSuccess) return GATO_ERR_CUDA;
        h->phi_pending = 0;
    }
    const size_t f = sizeof(float), K = (size_t)(w.N - 1);
    struct Item { float* dst; const float* src; size_t width, stride; } items[] = {
        {S_diag, w.D, (size_t)w.N * w.n * w.n, w.sNnn},
        {S_off, w.O, K * w.n * w.n, w.sKnn},
        {gamma, w.rhs[0].gamma, (size_t)w.N * w.n, w.sNn},
        {Phi_diag, w.Pd, (size_t)w.N * w.n * w.n, w.sNnn},
        {Phi_off, w.Po, K * w.n * w.n, w.sKnn},
    };
    for (const Item& it : items) {
        if (!it.dst || it.width == 0) continue;
        cudaError_t e = cudaMemcpy2DAsync(it.dst, it.width * f, it.src, it.stride * f,
                                          it.width * f, (size_t)w.M, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return GATO_ERR_CUDA;
    }
    return GATO_OK;
}

int gato_pcg_solve(gato_handle* h, const gato_params* p, const float* lambda0, float* lambda,
                   float* dX, float* dU, int32_t* iters, uint32_t* status, void* stream)
{
    if (!h || !params_valid(p) || !lambda || !dX || !iters || !status) return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && !dU) return GATO_ERR_INVALID_ARG;
    if (p->pcg_precision == GATO_PCG_PRECISION_FF &&
        !gato::pcg_ff_fits(h->w.N, h->w.n, (size_t)h->smem_optin))
        return GATO_ERR_UNSUPPORTED;
    h->w.status = status;
    cudaStream_t st = (cudaStream_t)stream;
    begin_timing(h, st);
    cudaError_t err = gato::launch_pcg(h, p, lambda0, lambda, dX, dU, iters, status, st);
    record(h, 2, st);
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return cuda_fail(err);
}

int gato_bdsv_solve(gato_handle* h, const gato_params* p, float* lambda, float* dX, float* dU,
                    int32_t* iters, uint32_t* status, void* stream)
{
    if (!h || !params_valid(p) || !lambda || !dX || !iters || !status)
        return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && !dU) return GATO_ERR_INVALID_ARG;
    const int ls = p->linsys == GATO_LINSYS_AUTO ? GATO_LINSYS_BDSV : p->linsys;
    if (ls == GATO_LINSYS_PCG) return GATO_ERR_INVALID_ARG;
    h->w.status = status;
    cudaStream_t st = (cudaStream_t)stream;
    begin_timing(h, st);
    cudaError_t err = gato::launch_bdsv_factor(h, ls, status, st);
    if (err == cudaSuccess)
        err = gato::launch_bdsv_solve(h, ls, 0, lambda, dX, dU, iters, 0, status, st);
    record(h, 2, st);
    return unsupported_or_fail(err);
}

int gato_linesearch(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                    const float* q, const float* r, const float* A, const float* B,
                    const float* e, const float* s0, const float* dX, const float* dU,
                    float* merit, int32_t* best, uint32_t* status, void* stream)
{
    if (!h || !params_valid(p) || !lq_ok(h, Q, R, q, r, A, B, e, s0) || !dX || !merit || !best ||
        !status)
        return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && !dU) return GATO_ERR_INVALID_ARG;
    h->w.status = status;
    cudaStream_t st = (cudaStream_t)stream;
    begin_timing(h, st);
    cudaError_t err =
        gato::launch_merit(h, p, Q, R, q, r, A, B, e, s0, dX, dU, merit, best, status, st);
    record(h, 4, st);
    return cuda_fail(err);
}

int gato_solve_kkt(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                   const float* q, const float* r, const float* A, const float* B,
                   const float* e, const float* s0, float* dX, float* dU, float* lambda,
                   int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                   void* stream)
{
    if (!h || !params_valid(p) || !lq_ok(h, Q, R, q, r, A, B, e, s0) || !dX || !lambda ||
        !iters || !merit || !best || !status)
        return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && !dU) return GATO_ERR_INVALID_ARG;
    if (!gato::sizes_supported(h->w, p, h->smem_optin)) return GATO_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (gato::parts_for(h, p, false) > 1) {
        h->ev_used[0] = 0;  // no stage timing for a call in parts
        return gato::run_parts(h, p, Q, R, q, r, A, B, e, s0, dX, dU, lambda, iters, merit,
                               best, status, st, false);
    }
    h->parts_last = 1;
    begin_timing(h, st);
    return unsupported_or_fail(gato::run_solve_kkt(h, p, Q, R, q, r, A, B, e, s0, dX, dU,
                                                   lambda, iters, merit, best, status, st));
}

int gato_apply_step(gato_handle* h, const gato_params* p, const int32_t* best, const float* dX,
                    const float* dU, float* X, float* U, void* stream)
{
    if (!h || !params_valid(p) || !best || !dX || !X) return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && (!dU || !U)) return GATO_ERR_INVALID_ARG;
    h->w.status = nullptr;
    return cuda_fail(gato::launch_apply_step(h, p, best, dX, dU, X, U, (cudaStream_t)stream));
}

int gato_sqp_linear(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                    const float* Q, const float* R, const float* q, const float* r,
                    const float* A, const float* B, const float* c, const float* xs, float* X,
                    float* U, float* lambda, float* rho, float* merit_hist, int32_t* iters_hist,
                    uint32_t* status, void* stream)
{
    if (!h || !params_valid(p) || !sqp_params_valid(sp) || !lq_ok(h, Q, R, q, r, A, B, c, xs) ||
        !X || !lambda || !rho || !merit_hist || !status)
        return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && !U) return GATO_ERR_INVALID_ARG;
    if (!gato::sizes_supported(h->w, p, h->smem_optin)) return GATO_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const SqpArgs a{Q, R, q, r, A, B, c, xs, X, U, lambda, rho, merit_hist, iters_hist, status};
    cudaError_t err = cudaMemsetAsync(h->w.sqpt, 0, sizeof(int) * h->w.M, st);
    if (err != cudaSuccess) return GATO_ERR_CUDA;
    if (!sp->use_graph) {
        for (int k = 0; k < sp->iters && err == cudaSuccess; ++k)
            err = sqp_iteration(h, p, sp, a, st);
        return unsupported_or_fail(err);
    }
    unsigned char key[sizeof(h->sqp_key)];
    sqp_key(key, h, p, sp, a);
    if (!h->sqp_exec || memcmp(key, h->sqp_key, sizeof(key)) != 0) {
        err = record_sqp_graph(h, p, sp, a);
        if (err != cudaSuccess) return unsupported_or_fail(err);
        memcpy(h->sqp_key, key, sizeof(key));
    }
    for (int k = 0; k < sp->iters && err == cudaSuccess; ++k)
        err = cudaGraphLaunch(h->sqp_exec, st);
    return unsupported_or_fail(err);
}

}  // extern "C"
