// gato_parts.cu -- the KKT solve of a batch as concurrent parts, from device
// buffers (gato_solve_kkt) or host buffers (gato_solve_kkt_host).  Not on the
// GATO pages; a GB300-side scheduling choice.
//
// The batch is split into parts of consecutive solves.  Each part has its own
// internal stream and its own sub-batch handle (workspace, work counters and
// merit counters), so the parts share no scratch and their kernels run
// concurrently: one part's formation, right-hand side and merit fill the SMs
// that another part's PCG leaves idle in its last wave.  From host buffers,
// part c also copies its slice of the inputs into device staging buffers
// first and its slice of the outputs back last, so the copies of one part
// overlap the kernels of the others.  A solve's arithmetic does not depend on
// its position in the batch, so the outputs do not depend on the part count.
#include <stdlib.h>
#include <string.h>

#include "gato_internal.cuh"

struct gato_parts {
    int nstreams;     // streams and events created (min(M, GATO_MAX_PARTS))
    int count_parts;  // parts of the current partition (0: none yet)
    int small_first;  // the current partition's first part is the short one
    int first[GATO_MAX_PARTS], count[GATO_MAX_PARTS];
    gato_handle sub[GATO_MAX_PARTS];  // views into the handle's workspace
    cudaStream_t st[GATO_MAX_PARTS];
    cudaEvent_t done[GATO_MAX_PARTS];
    // each part's low-priority side stream and its fork/join events
    cudaStream_t side[GATO_MAX_PARTS];
    cudaEvent_t fork[GATO_MAX_PARTS], join[GATO_MAX_PARTS];
    cudaEvent_t entry;
    void* dev;  // host entry: staging for the inputs and outputs of all M solves
    // per-solve sizes (elements) of the caller's arrays and, for the staging,
    // their offsets (bytes)
    size_t n_Q, n_R, n_q, n_r, n_A, n_B, n_e, n_s0, n_dX, n_dU, n_lam;
    size_t o_Q, o_R, o_q, o_r, o_A, o_B, o_e, o_s0, o_dX, o_dU, o_lam, o_merit, o_iters, o_best,
        o_status;
};

namespace gato {
namespace {

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

void release(gato_parts* pp)
{
    if (!pp) return;
    for (int c = 0; c < pp->nstreams; ++c) {
        if (pp->st[c]) cudaStreamDestroy(pp->st[c]);
        if (pp->done[c]) cudaEventDestroy(pp->done[c]);
        if (pp->side[c]) cudaStreamDestroy(pp->side[c]);
        if (pp->fork[c]) cudaEventDestroy(pp->fork[c]);
        if (pp->join[c]) cudaEventDestroy(pp->join[c]);
    }
    if (pp->entry) cudaEventDestroy(pp->entry);
    if (pp->dev) cudaFree(pp->dev);
    free(pp);
}

// the parts as views into the handle's workspace: part c takes the next
// 256-byte-aligned region of the size carve_workspace gives for its solves
// (the handle's allocation has room for any partition, see
// parts_extra_bytes); no allocation.  Equal parts, or with small_first and
// three parts or more a first part of about half the others' size (from host
// buffers nothing overlaps the first part's input copy, so it is kept short;
// with two parts the other part would carry three quarters of the batch)
void partition(gato_handle* h, int k, bool small_first)
{
    gato_parts* pp = h->pipe;
    const Work& w = h->w;
    const int c0 = (small_first && k > 2) ? (w.M / (2 * k) > 0 ? w.M / (2 * k) : 1) : 0;
    const int rest = w.M - c0, kr = c0 ? k - 1 : k;
    size_t off = 0;
    int first = 0;
    for (int c = 0; c < k; ++c) {
        const int r = c0 ? c - 1 : c;
        const int cnt = (c0 && c == 0) ? c0 : rest / kr + (r < rest % kr ? 1 : 0);
        pp->first[c] = first;
        pp->count[c] = cnt;
        first += cnt;
        gato_handle& sh = pp->sub[c];
        memset(&sh, 0, sizeof(sh));
        sh.device = h->device;
        sh.smem_optin = h->smem_optin;
        sh.num_sms = h->num_sms;
        sh.base = (char*)h->base + off;
        sh.bytes = carve_workspace(sh.w, cnt, w.N, w.n, w.m, nullptr);
        carve_workspace(sh.w, cnt, w.N, w.n, w.m, (float*)sh.base);
        sh.parts = 1;
        sh.batch_M = w.M;  // the parts run concurrently
        sh.side = pp->side[c];
        sh.ev_fork = pp->fork[c];
        sh.ev_join = pp->join[c];
        off += align256(sh.bytes);
    }
    pp->count_parts = k;
    pp->small_first = small_first ? 1 : 0;
}

// the host entry's device staging, allocated at its first use
int ensure_staging(gato_parts* pp, int M)
{
    if (pp->dev) return GATO_OK;
    const size_t f = sizeof(float), i4 = sizeof(int32_t);
    size_t off = 0;
    auto place = [&](size_t& o, size_t per_solve_bytes) {
        o = off;
        off += align256(per_solve_bytes * (size_t)M);
    };
    place(pp->o_Q, pp->n_Q * f);
    place(pp->o_R, pp->n_R * f);
    place(pp->o_q, pp->n_q * f);
    place(pp->o_r, pp->n_r * f);
    place(pp->o_A, pp->n_A * f);
    place(pp->o_B, pp->n_B * f);
    place(pp->o_e, pp->n_e * f);
    place(pp->o_s0, pp->n_s0 * f);
    place(pp->o_dX, pp->n_dX * f);
    place(pp->o_dU, pp->n_dU * f);
    place(pp->o_lam, pp->n_lam * f);
    place(pp->o_merit, (GATO_MAX_ALPHA + 1) * f);
    place(pp->o_iters, i4);
    place(pp->o_best, i4);
    place(pp->o_status, i4);
    if (cudaMalloc(&pp->dev, off) != cudaSuccess) {
        cudaGetLastError();
        pp->dev = nullptr;
        return GATO_ERR_NO_MEMORY;
    }
    return GATO_OK;
}

}  // namespace

// beyond the handle's own workspace, the parts need one work-counter block
// each, and each part's region starts on a 256-byte boundary
size_t parts_extra_bytes() { return (size_t)GATO_MAX_PARTS * 512; }

cudaError_t priority_stream_create(cudaStream_t* st, bool highest)
{
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e != cudaSuccess) return e;
    return cudaStreamCreateWithPriority(st, cudaStreamNonBlocking, highest ? greatest : least);
}

cudaError_t side_stream_create(cudaStream_t* st, cudaEvent_t* fork, cudaEvent_t* join)
{
    cudaError_t e = priority_stream_create(st, false);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(join, cudaEventDisableTiming);
    return e;
}

// streams and events for up to min(M, GATO_MAX_PARTS) parts, at gato_create
int parts_init(gato_handle* h)
{
    const Work& w = h->w;
    const size_t N = w.N, n = w.n, m = w.m, K = N - 1;
    gato_parts* pp = (gato_parts*)calloc(1, sizeof(gato_parts));
    if (!pp) return GATO_ERR_NO_MEMORY;
    pp->n_Q = N * n * n;
    pp->n_R = K * m * m;
    pp->n_q = N * n;
    pp->n_r = K * m;
    pp->n_A = K * n * n;
    pp->n_B = K * n * m;
    pp->n_e = K * n;
    pp->n_s0 = n;
    pp->n_dX = N * n;
    pp->n_dU = K * m;
    pp->n_lam = N * n;
    pp->nstreams = w.M < GATO_MAX_PARTS ? w.M : GATO_MAX_PARTS;
    int rc = GATO_OK;
    if (cudaEventCreateWithFlags(&pp->entry, cudaEventDisableTiming) != cudaSuccess)
        rc = GATO_ERR_CUDA;
    // the parts' own streams at the highest priority, so that the blocks of
    // their stages are dispatched before those of their side streams
    for (int c = 0; c < pp->nstreams && rc == GATO_OK; ++c)
        if (priority_stream_create(&pp->st[c], true) != cudaSuccess ||
            cudaEventCreateWithFlags(&pp->done[c], cudaEventDisableTiming) != cudaSuccess ||
            side_stream_create(&pp->side[c], &pp->fork[c], &pp->join[c]) != cudaSuccess)
            rc = GATO_ERR_CUDA;
    if (rc != GATO_OK) {
        release(pp);
        return rc;
    }
    h->pipe = pp;
    return GATO_OK;
}

// The caller's choice (capped at M), else by batch size and call: one part
// below 64 solves, two below 128, four from there (measured at N = 128 with
// PCG corrections: two parts gain 3-4% at 64-96 solves, four 1-4% from 128;
// below 64 one is best).  A call on device buffers whose corrections are
// direct after a PCG main solve already overlaps its longest short stage
// (the factorisation, on the side stream) with the PCG, and fewer parts do
// better there: one while the PCG holds the whole batch at once (one wave),
// two beyond (measured: 128 solves of N = 128 1.09 ms in one part against
// 1.18 in two, 152 1.20 against 1.21, 200 1.90 against 1.86, 256 1.97
// against 1.91; 256 of N = 64 1.01 against 1.07, of N = 32 0.64 against
// 0.73, of N = 16 0.39 against 0.47; 608 of N = 16 0.52 against 0.56; 128 of
// N = 16, n = 36 3.49 against 3.56 ms).  The host entry keeps the first
// rule: its parts also hide the input copies.
int parts_for(const gato_handle* h, const gato_params* p, bool host)
{
    const int M = h->w.M;
    int k = h->parts;
    if (k <= 0) {
        const bool forked = !host && p && p->refine_solver == GATO_REFINE_SOLVER_DIRECT &&
                            p->refine_steps > 0 && linsys_for(p, h->w.N) == GATO_LINSYS_PCG;
        k = forked ? (M > pcg_solves_per_wave(h, p) ? 2 : 1)
                   : (M >= 128 ? 4 : (M >= 64 ? 2 : 1));
    }
    if (k > M) k = M;
    return k;
}

void parts_free(gato_handle* h)
{
    if (!h) return;
    release(h->pipe);
    h->pipe = nullptr;
}

int run_parts(gato_handle* h, const gato_params* p, const float* Q, const float* R,
              const float* q, const float* r, const float* A, const float* B, const float* e,
              const float* s0, float* dX, float* dU, float* lambda, int32_t* iters, float* merit,
              int32_t* best, uint32_t* status, cudaStream_t user, bool host)
{
    const int k = parts_for(h, p, host);
    h->parts_last = k;
    gato_parts* pp = h->pipe;
    if (!pp || k > pp->nstreams) return GATO_ERR_INVALID_ARG;
    if (pp->count_parts != k || pp->small_first != (host ? 1 : 0)) partition(h, k, host);
    if (host) {
        const int rc = ensure_staging(pp, h->w.M);
        if (rc != GATO_OK) return rc;
    }
    char* dev = (char*)pp->dev;
    const size_t f = sizeof(float), i4 = sizeof(int32_t);
    const size_t A1 = (size_t)p->n_alpha + 1;  // merit row stride of the caller's array
    cudaError_t err = cudaEventRecord(pp->entry, user);
    for (int c = 0; c < k && err == cudaSuccess; ++c) {
        cudaStream_t st = pp->st[c];
        gato_handle* sh = &pp->sub[c];
        sh->pcg_kernel = h->pcg_kernel;
        sh->bdsv_kernel = h->bdsv_kernel;
        sh->force_smem_form = h->force_smem_form;
        sh->timing = 0;
        sh->pcg_ran = sh->refine_ran = 0;
        const size_t f0 = (size_t)pp->first[c], cnt = (size_t)pp->count[c];
        // the part's slice of an array with `per` elements of `es` bytes per
        // solve: in the staging (host entry) or in the caller's array
        auto part = [&](size_t o, size_t per, size_t es, const void* caller) {
            return host ? (void*)(dev + o + f0 * per * es)
                        : (caller ? (void*)((const char*)caller + f0 * per * es) : nullptr);
        };
        auto h2d = [&](size_t o, size_t per, size_t es, const void* src) {
            if (!host || err != cudaSuccess || per == 0) return;
            err = cudaMemcpyAsync(part(o, per, es, nullptr), (const char*)src + f0 * per * es,
                                  cnt * per * es, cudaMemcpyHostToDevice, st);
        };
        auto d2h = [&](size_t o, size_t per, size_t es, void* dst) {
            if (!host || err != cudaSuccess || per == 0) return;
            err = cudaMemcpyAsync((char*)dst + f0 * per * es, part(o, per, es, nullptr),
                                  cnt * per * es, cudaMemcpyDeviceToHost, st);
        };
        err = cudaStreamWaitEvent(st, pp->entry, 0);
        h2d(pp->o_Q, pp->n_Q, f, Q);
        h2d(pp->o_R, pp->n_R, f, R);
        h2d(pp->o_q, pp->n_q, f, q);
        h2d(pp->o_r, pp->n_r, f, r);
        h2d(pp->o_A, pp->n_A, f, A);
        h2d(pp->o_B, pp->n_B, f, B);
        h2d(pp->o_e, pp->n_e, f, e);
        h2d(pp->o_s0, pp->n_s0, f, s0);
        h2d(pp->o_status, 1, i4, status);
        if (err == cudaSuccess)
            err = run_solve_kkt(sh, p, (const float*)part(pp->o_Q, pp->n_Q, f, Q),
                                (const float*)part(pp->o_R, pp->n_R, f, R),
                                (const float*)part(pp->o_q, pp->n_q, f, q),
                                (const float*)part(pp->o_r, pp->n_r, f, r),
                                (const float*)part(pp->o_A, pp->n_A, f, A),
                                (const float*)part(pp->o_B, pp->n_B, f, B),
                                (const float*)part(pp->o_e, pp->n_e, f, e),
                                (const float*)part(pp->o_s0, pp->n_s0, f, s0),
                                (float*)part(pp->o_dX, pp->n_dX, f, dX),
                                (float*)part(pp->o_dU, pp->n_dU, f, dU),
                                (float*)part(pp->o_lam, pp->n_lam, f, lambda),
                                (int32_t*)part(pp->o_iters, 1, i4, iters),
                                (float*)part(pp->o_merit, A1, f, merit),
                                (int32_t*)part(pp->o_best, 1, i4, best),
                                (uint32_t*)part(pp->o_status, 1, i4, status), st);
        d2h(pp->o_dX, pp->n_dX, f, dX);
        d2h(pp->o_dU, pp->n_dU, f, dU);
        d2h(pp->o_lam, pp->n_lam, f, lambda);
        d2h(pp->o_iters, 1, i4, iters);
        d2h(pp->o_merit, A1, f, merit);
        d2h(pp->o_best, 1, i4, best);
        d2h(pp->o_status, 1, i4, status);
        // the caller's stream waits for whatever this part enqueued
        if (cudaEventRecord(pp->done[c], st) == cudaSuccess)
            cudaStreamWaitEvent(user, pp->done[c], 0);
    }
    // every part takes the same kernel (the choice counts the whole batch)
    if (err == cudaSuccess) {
        h->pcg_ran = pp->sub[k - 1].pcg_ran;
        h->refine_ran = pp->sub[k - 1].refine_ran;
    }
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GATO_OK : GATO_ERR_CUDA;
}

}  // namespace gato

extern "C" {

int gato_set_parts(gato_handle* h, int parts)
{
    if (!h || parts < 0 || parts > GATO_MAX_PARTS) return GATO_ERR_INVALID_ARG;
    h->parts = parts;
    return GATO_OK;
}

int gato_get_parts(const gato_handle* h, int* parts)
{
    if (!h || !parts) return GATO_ERR_INVALID_ARG;
    *parts = h->parts_last > 0 ? h->parts_last : gato::parts_for(h, nullptr, false);
    return GATO_OK;
}

int gato_solve_kkt_host(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                        const float* q, const float* r, const float* A, const float* B,
                        const float* e, const float* s0, float* dX, float* dU, float* lambda,
                        int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                        void* stream)
{
    using namespace gato;
    if (!h || !params_valid(p) || !Q || !q || !s0 || !dX || !lambda || !iters || !merit ||
        !best || !status)
        return GATO_ERR_INVALID_ARG;
    if (h->w.N > 1 && (!R || !r || !A || !B || !e || !dU)) return GATO_ERR_INVALID_ARG;
    if (!sizes_supported(h->w, p, h->smem_optin)) return GATO_ERR_UNSUPPORTED;
    h->ev_used[0] = 0;  // no stage timing for a call in parts
    return run_parts(h, p, Q, R, q, r, A, B, e, s0, dX, dU, lambda, iters, merit, best, status,
                     (cudaStream_t)stream, true);
}

}  // extern "C"
