// attnres_host.cu -- host-buffer training step of the read operator: the
// sources and dy live in host memory (pinned for full speed), the results go
// back to host memory, and the GPU work overlaps the transfers.
//
// The tokens are independent ("Fast Attention Residuals", section
// "Equation": normalisation and softmax run independently at each token), so
// the step runs over chunks of T tokens, double-buffered on the device, on
// three caller streams:
//   streams[1] (in):      H2D of chunk c's source rows and dy rows
//   streams[0] (compute): attnres_fwd + attnres_bwd of chunk c
//   streams[2] (out):     D2H of chunk c's y and dvalues rows
// so the copy into chunk c+1's buffer, the kernels of chunk c and the copy out
// of chunk c-1 run at the same time (H2D and D2H use separate copy engines).
// dq and dw_o are sums over all tokens: every chunk's backward writes its FP32
// sums into a row of its own, and the finalize kernel adds the rows in chunk
// order at the end (reproducible run to run).  Everything is enqueued
// asynchronously; streams[0] ends by waiting for the other two, so an event
// or synchronisation on streams[0] covers the whole step.
#include <cstring>

#include "attnres.h"
#include "kernels.cuh"

namespace attnres {
namespace {

struct HostStepLayout {
    size_t v, dv, dy, y, alpha, rstd, logit, o_rstd;  // offsets inside one buffer
    size_t buffer;                                     // bytes of one buffer
    size_t o_pre;                                      // FP32 [T, D] when the backward is not resident
    bool has_o_pre;
    size_t part, ws, dq, dw, dq32, dw32, qbuf, wbuf;   // offsets after the two buffers
    size_t total;
    int64_t chunks;
    size_t ws_bytes;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Chunk params for planning only: device rows of D elements; the pointers are
// placeholders (planning reads sizes, never memory).
attnres_params chunk_params(const attnres_params* p, int64_t T) {
    attnres_params c = *p;
    c.N = T;
    c.src_ld = p->D;
    for (int s = 0; s < p->S; ++s) c.src[s] = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    return c;
}

bool host_step_layout(const attnres_params* p, int64_t T, HostStepLayout* L) {
    const size_t S = static_cast<size_t>(p->S), D = static_cast<size_t>(p->D), R = static_cast<size_t>(p->R);
    const size_t t = static_cast<size_t>(T);
    size_t off = 0;
    L->v = off;
    off = up256(off + S * t * D * 2);
    L->dv = off;
    off = up256(off + S * t * D * 2);
    L->dy = off;
    off = up256(off + t * D * 2);
    L->y = off;
    off = up256(off + t * D * 2);
    L->alpha = off;
    off = up256(off + t * S * 4);
    L->rstd = off;
    off = up256(off + t * S * 4);
    L->logit = off;
    off = up256(off + t * S * 4);
    L->o_rstd = off;
    off = up256(off + t * 4);
    L->o_pre = off;
    {
        // the forward keeps FP32 o only when the backward cannot keep a
        // token's rows resident (the same rule as the Python binding)
        const attnres_params c = chunk_params(p, T);
        int64_t info[10];
        const bool resident = attnres_plan_info(&c, info) == ATTNRES_OK && info[5] != 0;
        L->has_o_pre = p->out_norm && !resident;
        if (L->has_o_pre) off = up256(off + t * D * 4);
    }
    L->buffer = off;
    L->chunks = (p->N + T - 1) / T;
    const size_t W = R + (p->out_norm ? D : 0);
    size_t o = 2 * L->buffer;
    L->part = o;
    o = up256(o + static_cast<size_t>(L->chunks) * W * 4);
    // the chunk backward's workspace (the same plan for every full chunk)
    const attnres_params c = chunk_params(p, T);
    L->ws_bytes = attnres_bwd_workspace_bytes(&c);
    L->ws = o;
    o = up256(o + L->ws_bytes);
    L->dq = o;  // bf16 [R]: per-chunk scratch, then the final dq
    o = up256(o + R * 2);
    L->dw = o;  // bf16 [D]
    o = up256(o + D * 2);
    L->dq32 = o;
    o = up256(o + R * 4);
    L->dw32 = o;
    o = up256(o + D * 4);
    L->qbuf = o;  // the query and the output-norm weight, copied in
    o = up256(o + R * 2);
    L->wbuf = o;
    o = up256(o + D * 2);
    L->total = o;
    return true;
}

}  // namespace
}  // namespace attnres

using namespace attnres;

extern "C" {

size_t attnres_step_host_workspace_bytes(const attnres_params* p, int64_t chunk_tokens) {
    if (!p || chunk_tokens < 1 || p->N < 0) return 0;
    HostStepLayout L;
    if (!host_step_layout(p, chunk_tokens, &L)) return 0;
    return L.total;
}

attnres_status attnres_step_host(const attnres_params* p, const void* q, const void* w_o, const void* dy,
                                 int64_t dy_ld, void* y, int64_t y_ld, void* const* dsrc, int64_t dsrc_ld,
                                 void* dq, float* dq_f32, void* dw_o, float* dw_o_f32, int64_t chunk_tokens,
                                 void* workspace, size_t workspace_bytes, void* const* streams) {
    if (!p || chunk_tokens < 1 || !streams) return ATTNRES_ERR_INVALID_ARG;
    const int64_t N = p->N;
    const size_t S = static_cast<size_t>(p->S), D = static_cast<size_t>(p->D), R = static_cast<size_t>(p->R);
    if (p->S < 1 || p->S > ATTNRES_MAX_S || p->D < 8 || p->D % 8 || p->R < 1 || p->R > p->D || N < 0)
        return ATTNRES_ERR_INVALID_ARG;
    if (!q || !dq || !dsrc || (p->out_norm && (!w_o || !dw_o))) return ATTNRES_ERR_INVALID_ARG;
    if (N == 0) {
        // empty sums: zero gradients of the query and the norm weight
        std::memset(dq, 0, R * 2);
        if (dq_f32) std::memset(dq_f32, 0, R * 4);
        if (p->out_norm) {
            std::memset(dw_o, 0, D * 2);
            if (dw_o_f32) std::memset(dw_o_f32, 0, D * 4);
        }
        return ATTNRES_OK;
    }
    if (!dy || !y || dy_ld < p->D || y_ld < p->D || dsrc_ld < p->D || p->src_ld < p->D)
        return ATTNRES_ERR_INVALID_ARG;
    for (int s = 0; s < p->S; ++s)
        if (!p->src[s] || !dsrc[s]) return ATTNRES_ERR_INVALID_ARG;
    const int64_t T = chunk_tokens < N ? chunk_tokens : N;
    HostStepLayout L;
    host_step_layout(p, T, &L);
    if (!workspace || workspace_bytes < L.total) return ATTNRES_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTNRES_ERR_ALIGNMENT;
    cudaStream_t cs = static_cast<cudaStream_t>(streams[0]);
    cudaStream_t is = static_cast<cudaStream_t>(streams[1]);
    cudaStream_t os = static_cast<cudaStream_t>(streams[2]);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const size_t W = R + (p->out_norm ? D : 0);

    cudaEvent_t ev[8];
    for (int i = 0; i < 8; ++i)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return ATTNRES_ERR_CUDA;
        }
    cudaEvent_t* in_ready = ev;       // [2]
    cudaEvent_t* out_ready = ev + 2;  // [2]
    cudaEvent_t* freed = ev + 4;      // [2]
    cudaEvent_t q_ready = ev[6], out_done = ev[7];
    attnres_status result = ATTNRES_OK;
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && result == ATTNRES_OK) result = ATTNRES_ERR_CUDA;
        return e == cudaSuccess;
    };

    uint16_t* qd = reinterpret_cast<uint16_t*>(ws + L.qbuf);
    uint16_t* wd = p->out_norm ? reinterpret_cast<uint16_t*>(ws + L.wbuf) : nullptr;
    ok(cudaMemcpyAsync(qd, q, R * 2, cudaMemcpyHostToDevice, is));
    if (wd) ok(cudaMemcpyAsync(wd, w_o, D * 2, cudaMemcpyHostToDevice, is));
    ok(cudaEventRecord(q_ready, is));
    ok(cudaStreamWaitEvent(cs, q_ready, 0));

    for (int64_t c = 0; c < L.chunks && result == ATTNRES_OK; ++c) {
        const int b = static_cast<int>(c & 1);
        unsigned char* buf = ws + static_cast<size_t>(b) * L.buffer;
        const int64_t n0 = c * T;
        const size_t nc = static_cast<size_t>(N - n0 < T ? N - n0 : T);
        unsigned char* vb = buf + L.v;
        unsigned char* dvb = buf + L.dv;
        // ---- in: the chunk's source rows and dy rows
        if (c >= 2) ok(cudaStreamWaitEvent(is, freed[b], 0));
        for (size_t s = 0; s < S; ++s)
            ok(cudaMemcpy2DAsync(vb + s * T * D * 2, D * 2,
                                 static_cast<const unsigned char*>(p->src[s]) + n0 * p->src_ld * 2,
                                 static_cast<size_t>(p->src_ld) * 2, D * 2, nc, cudaMemcpyHostToDevice, is));
        ok(cudaMemcpy2DAsync(buf + L.dy, D * 2, static_cast<const unsigned char*>(dy) + n0 * dy_ld * 2,
                             static_cast<size_t>(dy_ld) * 2, D * 2, nc, cudaMemcpyHostToDevice, is));
        ok(cudaEventRecord(in_ready[b], is));
        // ---- compute: forward and backward of the chunk
        ok(cudaStreamWaitEvent(cs, in_ready[b], 0));
        attnres_params pc = *p;
        pc.N = static_cast<int64_t>(nc);
        pc.src_ld = p->D;
        void* dptr[ATTNRES_MAX_S];
        for (size_t s = 0; s < S; ++s) {
            pc.src[s] = vb + s * T * D * 2;
            dptr[s] = dvb + s * T * D * 2;
        }
        float* alpha = reinterpret_cast<float*>(buf + L.alpha);
        float* rstd = reinterpret_cast<float*>(buf + L.rstd);
        float* logit = reinterpret_cast<float*>(buf + L.logit);
        float* o_rstd = p->out_norm ? reinterpret_cast<float*>(buf + L.o_rstd) : nullptr;
        float* o_pre = L.has_o_pre ? reinterpret_cast<float*>(buf + L.o_pre) : nullptr;
        attnres_status st2 = attnres_fwd(&pc, qd, wd, buf + L.y, alpha, rstd, logit, o_rstd, o_pre, cs);
        float* part = reinterpret_cast<float*>(ws + L.part) + static_cast<size_t>(c) * W;
        if (st2 == ATTNRES_OK)
            st2 = attnres_bwd(&pc, qd, wd, buf + L.dy, alpha, rstd, logit, o_rstd, o_pre, dptr, p->D,
                              ws + L.dq, part, p->out_norm ? ws + L.dw : nullptr,
                              p->out_norm ? part + R : nullptr, ws + L.ws, L.ws_bytes, cs);
        if (st2 != ATTNRES_OK) {
            result = st2;
            break;
        }
        ok(cudaEventRecord(out_ready[b], cs));
        // ---- out: y rows and dvalues rows back to the host
        ok(cudaStreamWaitEvent(os, out_ready[b], 0));
        ok(cudaMemcpy2DAsync(static_cast<unsigned char*>(y) + n0 * y_ld * 2, static_cast<size_t>(y_ld) * 2,
                             buf + L.y, D * 2, D * 2, nc, cudaMemcpyDeviceToHost, os));
        for (size_t s = 0; s < S; ++s)
            ok(cudaMemcpy2DAsync(static_cast<unsigned char*>(dsrc[s]) + n0 * dsrc_ld * 2,
                                 static_cast<size_t>(dsrc_ld) * 2, dvb + s * T * D * 2, D * 2, D * 2, nc,
                                 cudaMemcpyDeviceToHost, os));
        ok(cudaEventRecord(freed[b], os));
    }
    if (result == ATTNRES_OK) {
        // dq and dw_o: the chunks' FP32 sums added in chunk order
        uint16_t* dqd = reinterpret_cast<uint16_t*>(ws + L.dq);
        uint16_t* dwd = reinterpret_cast<uint16_t*>(ws + L.dw);
        float* dq32 = reinterpret_cast<float*>(ws + L.dq32);
        float* dw32 = reinterpret_cast<float*>(ws + L.dw32);
        ok(launch_finalize(reinterpret_cast<float*>(ws + L.part), static_cast<int>(L.chunks), p->R,
                           static_cast<int>(W), dqd, dq32, p->out_norm ? dwd : nullptr,
                           p->out_norm ? dw32 : nullptr, cs));
        ok(cudaMemcpyAsync(dq, dqd, R * 2, cudaMemcpyDeviceToHost, cs));
        if (dq_f32) ok(cudaMemcpyAsync(dq_f32, dq32, R * 4, cudaMemcpyDeviceToHost, cs));
        if (p->out_norm) {
            ok(cudaMemcpyAsync(dw_o, dwd, D * 2, cudaMemcpyDeviceToHost, cs));
            if (dw_o_f32) ok(cudaMemcpyAsync(dw_o_f32, dw32, D * 4, cudaMemcpyDeviceToHost, cs));
        }
    }
    // streams[0] covers the whole step
    ok(cudaEventRecord(out_done, os));
    ok(cudaStreamWaitEvent(cs, out_done, 0));
    for (int i = 0; i < 8; ++i) cudaEventDestroy(ev[i]);
    return result;
}

}  // extern "C"
