// kkt_host.cu -- kkt_solve on host buffers (kkt_solve_fwd_host): copies in, the kernel, copies out,
// pipelined over consecutive pieces of the token axis on three streams.  Declared in include/kkt.h.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "kkt_internal.cuh"
#include "kkt_test.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPieces = KKT_HOST_MAX_PIECES;
// a piece's inputs are copied in only once the outputs of the piece this many places earlier are
// back on the host, so that the inputs do not take the link from the outputs (the larger
// direction) early on
constexpr int kH2dAhead = 2;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The streams and events of one device: the copy-in and copy-out streams, and per piece the events
// "inputs in", "kernel done" and "outputs out", plus the call's start and end.  Created on the
// first call on the device and kept (cudaDeviceReset invalidates them).
struct DeviceQueues {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kMaxPieces] = {}, k_done[kMaxPieces] = {}, out_done[kMaxPieces] = {};
};
DeviceQueues g_queues[kMaxDevices];
std::mutex g_mutex;  // one enqueue at a time (the queues and events are shared)

int queues(int dev, DeviceQueues **out) {
    DeviceQueues &q = g_queues[dev];
    if (!q.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&q.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&q.out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&q.start, ef) != cudaSuccess || cudaEventCreateWithFlags(&q.end, ef) != cudaSuccess)
            return KKT_ERR_CUDA;
        for (int i = 0; i < kMaxPieces; ++i)
            if (cudaEventCreateWithFlags(&q.in_done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&q.k_done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&q.out_done[i], ef) != cudaSuccess)
                return KKT_ERR_CUDA;
        q.ready = true;
    }
    *out = &q;
    return KKT_OK;
}

// Bytes per (token, head) row of each tensor.
struct RowBytes {
    size_t k, v, beta, g, t, w, u;
};

RowBytes row_bytes(int dk, int dv, int C, int io_dtype, bool gated) {
    const size_t es = (io_dtype & ~KKT_T_OUT_F16) == KKT_IO_F32 ? 4 : 2;
    const size_t ts = (io_dtype & KKT_T_OUT_F16) ? 2 : 4;
    return RowBytes{es * dk, es * dv, 4, gated ? size_t(4) : size_t(0), ts * C, es * dk, es * dv};
}

// The workspace: the work counter, then the device copies (each 256-byte aligned), then the
// pieces' sequence offsets.
struct Layout {
    size_t counter, k, v, beta, g, t, w, u, cu, total;
};

Layout layout(int64_t ntok, int H, const RowBytes &rb, int nseq, int pieces) {
    Layout l{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    const size_t rows = size_t(ntok) * size_t(H);
    l.counter = take(KKT_WORKSPACE_BYTES);
    l.k = take(rows * rb.k);
    l.v = take(rows * rb.v);
    l.beta = take(rows * rb.beta);
    l.g = take(rows * rb.g);
    l.t = take(rows * rb.t);
    l.w = take(rows * rb.w);
    l.u = take(rows * rb.u);
    // every cut adds one sub-sequence, and every piece one offset more than it has sub-sequences
    l.cu = take(sizeof(int32_t) * size_t(nseq + 2 * pieces));
    l.total = off;
    return l;
}

// One piece: rows [n0, n1) of the flat token axis, its sub-sequences' offsets from n0 at
// cu[cu0 .. cu0 + nsub].
struct Piece {
    int64_t n0, n1;
    int cu0, nsub;
};

// Cuts the sequences [a_s, b_s) of the flat token axis into at most `parts` consecutive pieces of
// about equal token counts.  A sequence is cut only at a multiple of C from its start, so each
// piece's sub-sequences start at chunk boundaries and every chunk is one of the whole batch.  The
// last allowed piece takes everything left, so there are never more than `parts`.
void plan_pieces(const std::vector<int64_t> &starts, int C, int parts, std::vector<Piece> *out,
                 std::vector<int32_t> *cu) {
    const int64_t total = starts.back() - starts.front();
    if (total <= 0) return;
    int64_t target = (total + parts - 1) / parts;
    if (target < C) target = C;
    Piece cur{starts.front(), starts.front(), int(cu->size()), 0};
    cu->push_back(0);
    auto close = [&](int64_t at) {
        cur.n1 = at;
        out->push_back(cur);
        cur = Piece{at, at, int(cu->size()), 0};
        cu->push_back(0);
        if (int(out->size()) == parts - 1) target = INT64_MAX;  // the last piece takes the rest
    };
    if (parts == 1) target = INT64_MAX;
    for (size_t s = 0; s + 1 < starts.size(); ++s) {
        int64_t pos = starts[s];
        const int64_t end = starts[s + 1];
        while (pos < end) {
            const int64_t filled = pos - cur.n0;
            const int64_t room = target - filled;
            if (end - pos <= room) {  // the rest of the sequence fits
                cu->push_back(int32_t(end - cur.n0));
                ++cur.nsub;
                pos = end;
            } else if (room >= C) {  // take whole chunks up to the target, then close the piece
                const int64_t cut = pos + (room / C) * C;
                cu->push_back(int32_t(cut - cur.n0));
                ++cur.nsub;
                close(cut);
                pos = cut;
            } else if (filled > 0) {  // no room for a chunk: close the piece before this part
                close(pos);
            } else {  // an empty piece with target < C cannot happen (target >= C)
                cu->push_back(int32_t(end - cur.n0));
                ++cur.nsub;
                pos = end;
            }
        }
    }
    if (cur.nsub > 0) {
        cur.n1 = cur.n0 + (*cu)[cur.cu0 + cur.nsub];
        out->push_back(cur);
    } else {
        cu->pop_back();
    }
}

}  // namespace

extern "C" size_t kkt_host_workspace_bytes(int B, int T, int H, int dk, int dv, int C, int io_dtype, int gated,
                                           int varlen, int pieces) {
    if (B < 1 || T < 0 || H < 1 || pieces < 1 || pieces > kMaxPieces) return 0;
    const int64_t ntok = varlen ? int64_t(T) : int64_t(B) * T;
    return layout(ntok, H, row_bytes(dk, dv, C, io_dtype, gated != 0), B, pieces).total;
}

extern "C" int kkt_solve_fwd_host(const void *k, const void *v, const float *beta, const float *g,
                                  const int32_t *cu_seqlens, int B, int T, int H, int dk, int dv, int C,
                                  void *T_out, void *W_out, void *U_out, int io_dtype, int kernel, int pieces,
                                  void *workspace, size_t workspace_bytes, struct CUstream_st *stream) {
    if (!k || !v || !beta || !W_out || !U_out || !workspace) return KKT_ERR_ARG;
    if (B < 1 || T < 0 || H < 1 || pieces < 1 || pieces > kMaxPieces) return KKT_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KKT_ERR_ARG;
    const int sel = kkt_select_kernel(dk, dv, C, io_dtype, kernel);
    if (sel < 0) return -sel;
    const bool gated = g != nullptr;
    const int64_t ntok = cu_seqlens ? int64_t(T) : int64_t(B) * T;
    const RowBytes rb = row_bytes(dk, dv, C, io_dtype, gated);
    const Layout lo = layout(ntok, H, rb, B, pieces);
    if (workspace_bytes < lo.total) return KKT_ERR_ARG;
    // the sequences on the flat token axis (checked here: the offsets are host memory)
    std::vector<int64_t> starts(size_t(B) + 1);
    for (int s = 0; s <= B; ++s) starts[s] = cu_seqlens ? int64_t(cu_seqlens[s]) : int64_t(s) * T;
    if (starts[0] != 0 || starts[B] != ntok) return KKT_ERR_SEQLENS;
    for (int s = 0; s < B; ++s)
        if (starts[s + 1] < starts[s]) return KKT_ERR_SEQLENS;
    if (ntok == 0) return KKT_OK;
    std::vector<Piece> plan;
    std::vector<int32_t> cu;
    plan_pieces(starts, C, pieces, &plan, &cu);
    if (plan.empty() || int(plan.size()) > pieces || cu.size() * sizeof(int32_t) > lo.total - lo.cu)
        return KKT_ERR_ARG;  // cannot happen: the planner keeps to both bounds

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KKT_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> hold(g_mutex);
    DeviceQueues *q = nullptr;
    int st = queues(dev, &q);
    if (st != KKT_OK) return st;
    cudaStream_t main = reinterpret_cast<cudaStream_t>(stream);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t hrow = size_t(H);
    // the call starts after the work already on the caller's stream; the counter is cleared first
    if (!ok(cudaMemsetAsync(ws + lo.counter, 0, KKT_WORKSPACE_BYTES, main)) || !ok(cudaEventRecord(q->start, main)) ||
        !ok(cudaStreamWaitEvent(q->in, q->start, 0)) || !ok(cudaStreamWaitEvent(q->out, q->start, 0)))
        return KKT_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(ws + lo.cu, cu.data(), cu.size() * sizeof(int32_t), cudaMemcpyHostToDevice, q->in)))
        return KKT_ERR_CUDA;
    struct Tensor {
        const void *host;
        size_t dev_off, row;
    };
    const Tensor ins[4] = {{k, lo.k, rb.k}, {v, lo.v, rb.v}, {beta, lo.beta, rb.beta}, {g, lo.g, rb.g}};
    const Tensor outs[3] = {{T_out, lo.t, rb.t}, {W_out, lo.w, rb.w}, {U_out, lo.u, rb.u}};
    for (size_t p = 0; p < plan.size(); ++p) {
        const Piece &pc = plan[p];
        const size_t r0 = size_t(pc.n0) * hrow, nr = size_t(pc.n1 - pc.n0) * hrow;
        if (p >= size_t(kH2dAhead) && !ok(cudaStreamWaitEvent(q->in, q->out_done[p - kH2dAhead], 0)))
            return KKT_ERR_CUDA;
        for (const Tensor &t : ins) {
            if (!t.host || t.row == 0) continue;
            if (!ok(cudaMemcpyAsync(ws + t.dev_off + r0 * t.row, static_cast<const uint8_t *>(t.host) + r0 * t.row,
                                    nr * t.row, cudaMemcpyHostToDevice, q->in)))
                return KKT_ERR_CUDA;
        }
        if (!ok(cudaEventRecord(q->in_done[p], q->in)) || !ok(cudaStreamWaitEvent(main, q->in_done[p], 0)))
            return KKT_ERR_CUDA;
        // the piece: a packed batch of its sub-sequences, with its own offsets
        kkt::Problem pb;
        int which = 0;
        bool empty = false;
        st = kkt::make_problem(ws + lo.k + r0 * rb.k, ws + lo.v + r0 * rb.v,
                               reinterpret_cast<const float *>(ws + lo.beta + r0 * rb.beta),
                               gated ? reinterpret_cast<const float *>(ws + lo.g + r0 * rb.g) : nullptr,
                               reinterpret_cast<const int32_t *>(ws + lo.cu) + pc.cu0, pc.nsub, int(pc.n1 - pc.n0), H,
                               dk, dv, C, T_out ? ws + lo.t + r0 * rb.t : nullptr, ws + lo.w + r0 * rb.w,
                               ws + lo.u + r0 * rb.u, io_dtype, kernel, stream, &pb, &which, &empty);
        if (st != KKT_OK) return st;
        if (!empty) {
            if (which == KKT_KERNEL_TC) pb.tile_counter = reinterpret_cast<unsigned long long *>(ws + lo.counter);
            st = which == KKT_KERNEL_TC ? kkt::launch_tc(pb) : kkt::launch_simt(pb);
            if (st != KKT_OK) return st;
        }
        if (!ok(cudaEventRecord(q->k_done[p], main)) || !ok(cudaStreamWaitEvent(q->out, q->k_done[p], 0)))
            return KKT_ERR_CUDA;
        for (const Tensor &t : outs) {
            if (!t.host) continue;
            if (!ok(cudaMemcpyAsync(static_cast<uint8_t *>(const_cast<void *>(t.host)) + r0 * t.row,
                                    ws + t.dev_off + r0 * t.row, nr * t.row, cudaMemcpyDeviceToHost, q->out)))
                return KKT_ERR_CUDA;
        }
        if (!ok(cudaEventRecord(q->out_done[p], q->out))) return KKT_ERR_CUDA;
    }
    // the work enqueued on the caller's stream after this call runs after the copies out
    if (!ok(cudaEventRecord(q->end, q->out)) || !ok(cudaStreamWaitEvent(main, q->end, 0))) return KKT_ERR_CUDA;
    return KKT_OK;
}

// Test hook (kkt_test.h): the piece plan, host only.
extern "C" int kkt_test_plan_pieces(const int64_t *starts, int nseq, int C, int parts, int64_t *bounds, int32_t *nsub,
                                    int max_pieces, int32_t *cu, int cu_cap) {
    if (!starts || nseq < 1 || C < 1 || parts < 1 || !bounds || !nsub || !cu) return -1;
    std::vector<int64_t> st(starts, starts + nseq + 1);
    for (int s = 0; s < nseq; ++s)
        if (st[s + 1] < st[s]) return -1;
    std::vector<Piece> plan;
    std::vector<int32_t> offs;
    plan_pieces(st, C, parts, &plan, &offs);
    if (int(plan.size()) > max_pieces || int(offs.size()) > cu_cap) return -1;
    for (size_t p = 0; p < plan.size(); ++p) {
        bounds[2 * p] = plan[p].n0;
        bounds[2 * p + 1] = plan[p].n1;
        nsub[p] = plan[p].nsub;
    }
    std::memcpy(cu, offs.data(), offs.size() * sizeof(int32_t));
    return int(plan.size());
}
