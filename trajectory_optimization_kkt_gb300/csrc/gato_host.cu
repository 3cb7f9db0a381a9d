// gato_host.cu -- gato_solve_kkt_host: the KKT solve of a batch that lives in
// host memory.  Not on the GATO pages; it serves a host-resident batch on a
// GPU attached through a fast chip-to-chip link, where copying the whole
// batch in, solving and copying it out one after the other leaves the copy
// engines and the SMs idle in turn.
//
// The batch is split into parts of consecutive solves.  Each part has its own
// internal stream and its own sub-batch handle (workspace, work counters and
// merit counters), so the parts share no scratch: part c copies its slice of
// the inputs into device staging buffers, runs the same KKT core as
// gato_solve_kkt on its sub-batch handle, and copies its slice of the outputs
// back.  The copies of one part overlap the kernels of the others.  A solve's
// arithmetic does not depend on its position in the batch, so the outputs are
// those of gato_solve_kkt.
#include <stdlib.h>
#include <string.h>

#include "gato_internal.cuh"

struct gato_host_pipe {
    int chunks;
    int first[GATO_HOST_MAX_CHUNKS], count[GATO_HOST_MAX_CHUNKS];
    gato_handle* sub[GATO_HOST_MAX_CHUNKS];
    cudaStream_t st[GATO_HOST_MAX_CHUNKS];
    cudaEvent_t done[GATO_HOST_MAX_CHUNKS];
    cudaEvent_t entry;
    void* dev;  // device staging: the inputs and outputs of all M solves
    // per-solve sizes (elements) and offsets (bytes) of the staged arrays
    size_t n_Q, n_R, n_q, n_r, n_A, n_B, n_e, n_s0, n_dX, n_dU, n_lam, n_merit;
    size_t o_Q, o_R, o_q, o_r, o_A, o_B, o_e, o_s0, o_dX, o_dU, o_lam, o_merit, o_iters, o_best,
        o_status;
};

namespace gato {
namespace {

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

// parts for a batch of M solves: one per 64 solves, between 1 and 4, or the
// caller's choice (capped at M)
int chunk_count(const gato_handle* h)
{
    const int M = h->w.M;
    int k = h->host_chunks;
    if (k <= 0) {
        k = M / 64;
        if (k > 4) k = 4;
        if (k < 1) k = 1;
    }
    if (k > M) k = M;
    return k;
}

void pipe_release(gato_host_pipe* pp)
{
    if (!pp) return;
    for (int c = 0; c < pp->chunks; ++c) {
        if (pp->sub[c]) gato_destroy(pp->sub[c]);
        if (pp->st[c]) cudaStreamDestroy(pp->st[c]);
        if (pp->done[c]) cudaEventDestroy(pp->done[c]);
    }
    if (pp->entry) cudaEventDestroy(pp->entry);
    if (pp->dev) cudaFree(pp->dev);
    free(pp);
}

// a pipe of k parts for the handle's sizes; NO_MEMORY / CUDA on failure
int pipe_create(const gato_handle* h, int k, gato_host_pipe** out)
{
    const Work& w = h->w;
    const size_t M = w.M, N = w.N, n = w.n, m = w.m, K = N - 1;
    gato_host_pipe* pp = (gato_host_pipe*)calloc(1, sizeof(gato_host_pipe));
    if (!pp) return GATO_ERR_NO_MEMORY;
    pp->chunks = k;
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
    pp->n_merit = GATO_MAX_ALPHA + 1;
    size_t off = 0;
    auto place = [&](size_t& o, size_t per_solve_bytes) {
        o = off;
        off += align256(per_solve_bytes * M);
    };
    const size_t f = sizeof(float), i4 = sizeof(int32_t);
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
    place(pp->o_merit, pp->n_merit * f);
    place(pp->o_iters, i4);
    place(pp->o_best, i4);
    place(pp->o_status, i4);
    int rc = GATO_OK;
    if (cudaMalloc(&pp->dev, off) != cudaSuccess) {
        cudaGetLastError();
        pp->dev = nullptr;
        rc = GATO_ERR_NO_MEMORY;
    }
    if (rc == GATO_OK && cudaEventCreateWithFlags(&pp->entry, cudaEventDisableTiming) != cudaSuccess)
        rc = GATO_ERR_CUDA;
    int first = 0;
    for (int c = 0; c < k && rc == GATO_OK; ++c) {
        const int cnt = (int)(M / k) + (c < (int)(M % k) ? 1 : 0);
        pp->first[c] = first;
        pp->count[c] = cnt;
        first += cnt;
        if (cudaStreamCreateWithFlags(&pp->st[c], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&pp->done[c], cudaEventDisableTiming) != cudaSuccess) {
            rc = GATO_ERR_CUDA;
            break;
        }
        rc = gato_create(&pp->sub[c], cnt, w.N, w.n, w.m);
    }
    if (rc != GATO_OK) {
        pipe_release(pp);
        return rc;
    }
    *out = pp;
    return GATO_OK;
}

}  // namespace

void host_pipe_free(gato_handle* h)
{
    if (!h) return;
    pipe_release(h->pipe);
    h->pipe = nullptr;
}

}  // namespace gato

extern "C" {

int gato_set_host_chunks(gato_handle* h, int chunks)
{
    if (!h || chunks < 0 || chunks > GATO_HOST_MAX_CHUNKS) return GATO_ERR_INVALID_ARG;
    h->host_chunks = chunks;
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
    const int k = chunk_count(h);
    if (h->pipe && h->pipe->chunks != k) host_pipe_free(h);
    if (!h->pipe) {
        const int rc = pipe_create(h, k, &h->pipe);
        if (rc != GATO_OK) return rc;
    }
    gato_host_pipe* pp = h->pipe;
    cudaStream_t user = (cudaStream_t)stream;
    char* dev = (char*)pp->dev;
    const size_t f = sizeof(float), i4 = sizeof(int32_t);
    const size_t A1 = (size_t)p->n_alpha + 1;  // merit row stride of the caller's array
    cudaError_t err = cudaEventRecord(pp->entry, user);
    for (int c = 0; c < k && err == cudaSuccess; ++c) {
        cudaStream_t st = pp->st[c];
        gato_handle* sh = pp->sub[c];
        sh->pcg_kernel = h->pcg_kernel;
        sh->bdsv_kernel = h->bdsv_kernel;
        sh->force_smem_form = h->force_smem_form;
        sh->timing = 0;
        const size_t f0 = (size_t)pp->first[c], cnt = (size_t)pp->count[c];
        // the part's slice of a staged array (per: elements per solve)
        auto dptr = [&](size_t o, size_t per, size_t es) {
            return (void*)(dev + o + f0 * per * es);
        };
        auto h2d = [&](size_t o, size_t per, size_t es, const void* src) {
            if (err != cudaSuccess || per == 0) return;
            err = cudaMemcpyAsync(dptr(o, per, es), (const char*)src + f0 * per * es,
                                  cnt * per * es, cudaMemcpyHostToDevice, st);
        };
        auto d2h = [&](size_t o, size_t per, size_t es, void* dst) {
            if (err != cudaSuccess || per == 0) return;
            err = cudaMemcpyAsync((char*)dst + f0 * per * es, dptr(o, per, es), cnt * per * es,
                                  cudaMemcpyDeviceToHost, st);
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
            err = run_solve_kkt(
                sh, p, (const float*)dptr(pp->o_Q, pp->n_Q, f),
                (const float*)dptr(pp->o_R, pp->n_R, f), (const float*)dptr(pp->o_q, pp->n_q, f),
                (const float*)dptr(pp->o_r, pp->n_r, f), (const float*)dptr(pp->o_A, pp->n_A, f),
                (const float*)dptr(pp->o_B, pp->n_B, f), (const float*)dptr(pp->o_e, pp->n_e, f),
                (const float*)dptr(pp->o_s0, pp->n_s0, f), (float*)dptr(pp->o_dX, pp->n_dX, f),
                (float*)dptr(pp->o_dU, pp->n_dU, f), (float*)dptr(pp->o_lam, pp->n_lam, f),
                (int32_t*)dptr(pp->o_iters, 1, i4), (float*)dptr(pp->o_merit, A1, f),
                (int32_t*)dptr(pp->o_best, 1, i4), (uint32_t*)dptr(pp->o_status, 1, i4), st);
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
    if (err == cudaErrorInvalidConfiguration) return GATO_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GATO_OK : GATO_ERR_CUDA;
}

}  // extern "C"
