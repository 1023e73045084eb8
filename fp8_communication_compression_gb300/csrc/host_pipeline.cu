// The two-shot local path between host buffers, overlapped: the runtime
// behind taco_host_pipeline_run.
//
// The rows are split into C chunks.  For chunk c, one 2-D copy gathers the
// chunk's rows of all P shards from the host tensor [P][rows][d] into a
// device slot [P][Rc][d] (stream 0); compress, shard reduce and decompress
// run on stream 1; the result is copied back into the host output (stream
// 2).  Copies in, kernels and copies out of different chunks therefore run
// at the same time, and host-to-device and device-to-host copies use the
// two copy engines concurrently.
//
// Chaining: a call's copy into slot c waits only until the previous call's
// compress has consumed slot c, and its decompress into slot c only until
// the previous call's copy-out of slot c has finished, so consecutive calls
// overlap chunk by chunk.  The first call is ordered after the work already
// queued on the caller's stream; every call makes the caller's stream wait
// for its last copy-out.
//
// The pipeline owns only CUDA streams and events; every device byte it uses
// is the caller's workspace, carved into C equal chunk slots.

#include <cstdint>
#include <new>

#include "internal.h"

namespace taco {

namespace {

constexpr int kMaxChunks = 64;
constexpr uint64_t kAlign = 256;

uint64_t round_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

}  // namespace

struct HostPipeline {
    int P = 0;
    int64_t rows = 0, d = 0, R = 0;  // R: rows per chunk (the last chunk may hold fewer)
    int block = 0, C = 0;
    bool out_bf16 = false;
    int device = -1;
    bool started = false;
    // offsets of the buffers inside one chunk slot, and the slot size
    uint64_t o_x = 0, o_codes = 0, o_alpha = 0, o_scale = 0, o_rcodes = 0, o_ralpha = 0, o_rscale = 0, o_out = 0;
    uint64_t slot = 0;
    cudaStream_t s[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t ev_in[kMaxChunks] = {}, ev_comp[kMaxChunks] = {}, ev_done[kMaxChunks] = {},
                ev_out[kMaxChunks] = {};
    cudaEvent_t ev_entry = nullptr, ev_exit = nullptr;
};

int host_pipeline_max_chunks() { return kMaxChunks; }

static void release(HostPipeline *p)
{
    for (int c = 0; c < kMaxChunks; ++c) {
        for (cudaEvent_t e : {p->ev_in[c], p->ev_comp[c], p->ev_done[c], p->ev_out[c]})
            if (e)
                cudaEventDestroy(e);
    }
    if (p->ev_entry)
        cudaEventDestroy(p->ev_entry);
    if (p->ev_exit)
        cudaEventDestroy(p->ev_exit);
    for (cudaStream_t st : p->s)
        if (st)
            cudaStreamDestroy(st);
    delete p;
}

cudaError_t host_pipeline_create(int P, int64_t rows, int64_t d, int block, int chunks, bool out_bf16,
                                 HostPipeline **out, uint64_t *workspace_bytes)
{
    HostPipeline *p = new (std::nothrow) HostPipeline;
    if (!p)
        return cudaErrorMemoryAllocation;
    p->P = P;
    p->rows = rows;
    p->d = d;
    p->block = block;
    p->R = (rows + chunks - 1) / chunks;
    p->C = static_cast<int>((rows + p->R - 1) / p->R);
    p->out_bf16 = out_bf16;
    const uint64_t e = static_cast<uint64_t>(p->R) * d, nb = e / block;
    uint64_t off = 0;
    auto take = [&](uint64_t bytes) {
        const uint64_t o = off;
        off = round_up(off + bytes);
        return o;
    };
    p->o_x = take(2 * P * e);
    p->o_codes = take(P * e);
    p->o_alpha = take(4 * P * nb);
    p->o_scale = take(4 * P * nb);
    p->o_rcodes = take(e);
    p->o_ralpha = take(4 * nb);
    p->o_rscale = take(4 * nb);
    p->o_out = take((out_bf16 ? 2 : 4) * e);
    p->slot = off;

    cudaError_t err = cudaGetDevice(&p->device);
    for (int i = 0; i < 3 && err == cudaSuccess; ++i)
        err = cudaStreamCreateWithFlags(&p->s[i], cudaStreamNonBlocking);
    for (int c = 0; c < p->C && err == cudaSuccess; ++c) {
        for (cudaEvent_t *ev : {&p->ev_in[c], &p->ev_comp[c], &p->ev_done[c], &p->ev_out[c]})
            if (err == cudaSuccess)
                err = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    }
    if (err == cudaSuccess)
        err = cudaEventCreateWithFlags(&p->ev_entry, cudaEventDisableTiming);
    if (err == cudaSuccess)
        err = cudaEventCreateWithFlags(&p->ev_exit, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        release(p);
        return err;
    }
    *out = p;
    *workspace_bytes = p->slot * p->C;
    return cudaSuccess;
}

void host_pipeline_destroy(HostPipeline *p)
{
    if (p)
        release(p);
}

int host_pipeline_device(const HostPipeline *p) { return p->device; }

uint64_t host_pipeline_workspace(const HostPipeline *p) { return p->slot * p->C; }

cudaError_t host_pipeline_run(HostPipeline *p, const void *x_host, void *out_host, void *workspace, float e_target,
                              float eps, cudaStream_t stream)
{
    cudaError_t err = cudaSuccess;
    if (!p->started) {
        if ((err = cudaEventRecord(p->ev_entry, stream)) != cudaSuccess)
            return err;
        for (cudaStream_t st : p->s)
            if ((err = cudaStreamWaitEvent(st, p->ev_entry, 0)) != cudaSuccess)
                return err;
    }
    const int P = p->P, block = p->block;
    const int64_t d = p->d;
    const size_t out_elem = p->out_bf16 ? 2 : 4;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    for (int c = 0; c < p->C; ++c) {
        const int64_t r0 = c * p->R, Rc = (p->rows - r0 < p->R) ? p->rows - r0 : p->R;
        const int64_t e = Rc * d, nb = e / block;
        uint8_t *slot = ws + c * p->slot;
        auto *x = reinterpret_cast<uint16_t *>(slot + p->o_x);
        auto *codes = slot + p->o_codes;
        auto *alpha = reinterpret_cast<float *>(slot + p->o_alpha);
        auto *scale = reinterpret_cast<float *>(slot + p->o_scale);
        auto *rcodes = slot + p->o_rcodes;
        auto *ralpha = reinterpret_cast<float *>(slot + p->o_ralpha);
        auto *rscale = reinterpret_cast<float *>(slot + p->o_rscale);
        void *out = slot + p->o_out;

        // copy in: the chunk's rows of every shard, one 2-D copy
        if (p->started && (err = cudaStreamWaitEvent(p->s[0], p->ev_comp[c], 0)) != cudaSuccess)
            return err;
        const auto *src = static_cast<const uint8_t *>(x_host) + static_cast<size_t>(r0 * d) * 2;
        if ((err = cudaMemcpy2DAsync(x, static_cast<size_t>(e) * 2, src, static_cast<size_t>(p->rows * d) * 2,
                                     static_cast<size_t>(e) * 2, static_cast<size_t>(P), cudaMemcpyHostToDevice,
                                     p->s[0])) != cudaSuccess ||
            (err = cudaEventRecord(p->ev_in[c], p->s[0])) != cudaSuccess)
            return err;

        // compress all shards of the chunk, reduce them, decompress the result
        if ((err = cudaStreamWaitEvent(p->s[1], p->ev_in[c], 0)) != cudaSuccess ||
            (err = launch_compress(x, P * e / 128, block, e_target, eps, codes, alpha, scale, false, p->s[1])) !=
                cudaSuccess ||
            (err = cudaEventRecord(p->ev_comp[c], p->s[1])) != cudaSuccess)
            return err;
        ShardPtrs sp = {};
        for (int q = 0; q < P; ++q) {
            sp.codes[q] = codes + q * e;
            sp.alpha[q] = alpha + q * nb;
            sp.scale[q] = scale + q * nb;
        }
        if ((err = launch_taco_reduce(P, sp, nb, block, e_target, eps, rcodes, ralpha, rscale, p->s[1])) !=
            cudaSuccess)
            return err;
        if (p->started && (err = cudaStreamWaitEvent(p->s[1], p->ev_out[c], 0)) != cudaSuccess)
            return err;
        if ((err = launch_decompress(rcodes, ralpha, rscale, e / 128, block, out, p->out_bf16, false, p->s[1])) !=
                cudaSuccess ||
            (err = cudaEventRecord(p->ev_done[c], p->s[1])) != cudaSuccess)
            return err;

        // copy out
        auto *dst = static_cast<uint8_t *>(out_host) + static_cast<size_t>(r0 * d) * out_elem;
        if ((err = cudaStreamWaitEvent(p->s[2], p->ev_done[c], 0)) != cudaSuccess ||
            (err = cudaMemcpyAsync(dst, out, static_cast<size_t>(e) * out_elem, cudaMemcpyDeviceToHost,
                                   p->s[2])) != cudaSuccess ||
            (err = cudaEventRecord(p->ev_out[c], p->s[2])) != cudaSuccess)
            return err;
    }
    p->started = true;
    if ((err = cudaEventRecord(p->ev_exit, p->s[2])) != cudaSuccess)
        return err;
    return cudaStreamWaitEvent(stream, p->ev_exit, 0);
}

}  // namespace taco
