// Kimi Context Parallel (KCP) forward, simulated on one device.
//
// Page "flash-linear-attention KCP precision-debugging guide" (sections
// "背景：KCP 调试的特殊性", "h与dh的跨 rank 语义", "调试脚本布局：搭建单设备
// KCP 模拟器"): the packed token range is cut into world_size contiguous rank
// slices; each rank processes its local pieces of the sequences.  Only the
// first local piece of a rank can continue a sequence from the previous rank,
// and only the last local piece can continue into the next one.  Per rank,
//   pre-process: for the last local piece, the transition M_r and the
//                zero-start state S_ext,r, so that the state leaving the rank
//                is  M_r S_start + S_ext,r;
//   merge:       the state entering rank r + 1 is that expression evaluated
//                with S_start = the state entering rank r (when the piece is
//                a continuation) or the sequence's own initial state;
//   forward:     the local chunked forward with the merged state as the
//                initial state of the first local piece.
// The ranks are simulated by looping over them on one stream; every step runs
// in this library's kernels (the forward's prep + scan kernels and the merge
// kernel below).  M_r comes from the forward itself: with v = 0 the
// recurrence is linear in the state with no source term, so starting from the
// identity it ends at M_r (in the [V, K] layout, M_r^T).
#include <cstdint>
#include <vector>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr size_t STATE_BYTES = (size_t)VD * KD * 4;   // one [V, K] fp32 state

// out[h] = S[h] Mt[h] + E[h] for 128 x 128 fp32 matrices in the [V, K]
// layout (S = null means a zero start: out = E).  One CTA per head, 256
// threads, an 8 x 8 block of outputs per thread, K staged in 16-wide slabs.
__global__ void __launch_bounds__(256) kda_kcp_merge_kernel(const float* S, const float* Mt, const float* E,
                                                            float* out) {
    __shared__ float sA[128][17];
    __shared__ float sB[16][128];
    const size_t off = (size_t)blockIdx.x * VD * KD;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = E[off + (size_t)(ty * 8 + i) * KD + tx * 8 + j];
    if (S != nullptr) {
        for (int j0 = 0; j0 < KD; j0 += 16) {
            for (int e = threadIdx.x; e < 128 * 16; e += 256) {
                sA[e >> 4][e & 15] = S[off + (size_t)(e >> 4) * KD + j0 + (e & 15)];
                sB[e >> 7][e & 127] = Mt[off + (size_t)(j0 + (e >> 7)) * KD + (e & 127)];
            }
            __syncthreads();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                float a[8], b[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = sA[ty * 8 + i][jj];
#pragma unroll
                for (int j = 0; j < 8; ++j) b[j] = sB[jj][tx * 8 + j];
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) out[off + (size_t)(ty * 8 + i) * KD + tx * 8 + j] = acc[i][j];
}

// H identity states ([V, K] layout).
__global__ void kda_kcp_identity_kernel(float* I, int H) {
    const size_t n = (size_t)H * VD * KD;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const int kk = (int)(e % KD), vv = (int)((e / KD) % VD);
        I[e] = vv == kk ? 1.f : 0.f;
    }
}

struct Piece {
    int n;          // sequence
    long long a, b; // packed token range [a, b)
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Rank r owns packed tokens [T r / W, T (r + 1) / W).
long long rank_start(long long T, int r, int W) { return T * r / W; }

struct Layout {
    size_t fwd, vzero, ident, mt, ext, sin, h0l, htl, scratch_o, cu, total;
    long long tmax;
};

Layout layout(int T, int H, int N, int W) {
    Layout L{};
    long long tmax = 0;
    for (int r = 0; r < W; ++r) {
        const long long len = rank_start(T, r + 1, W) - rank_start(T, r, W);
        tmax = len > tmax ? len : tmax;
    }
    L.tmax = tmax;
    const int tf = (int)(tmax > 0 ? tmax : 1);
    size_t o = 0;
    L.fwd = o;
    o += align256(kda_fwd_workspace_bytes(1, tf, H, KD, VD, N));
    const size_t tok_bytes = (size_t)tf * H * VD * 2;
    L.vzero = o;
    o += align256(tok_bytes);
    L.scratch_o = o;
    o += align256(tok_bytes);
    const size_t hs = (size_t)H * STATE_BYTES;
    L.ident = o;
    o += hs;
    L.mt = o;
    o += (size_t)W * hs;
    L.ext = o;
    o += (size_t)W * hs;
    L.sin = o;
    o += (size_t)W * hs;
    L.h0l = o;
    o += (size_t)N * hs;
    L.htl = o;
    o += (size_t)N * hs;
    L.cu = o;
    o += align256((size_t)W * (N + 1 + 2) * sizeof(int32_t));
    L.total = o;
    return L;
}

}  // namespace

}  // namespace kda

extern "C" size_t kda_kcp_workspace_bytes(int T, int H, int K, int V, int N, int world_size) {
    if (T < 0 || H < 1 || N < 1 || world_size < 1 || world_size > 4096 || K != kda::KD || V != kda::VD) return 0;
    return kda::layout(T, H, N, world_size).total;
}

extern "C" kda_status kda_kcp_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  float scale, const float* h0, const int32_t* cu_seqlens_host, void* o, float* ht,
                                  int T, int H, int K, int V, int N, int world_size, unsigned flags, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    using namespace kda;
    if (K != KD || V != VD) return KDA_ERR_UNSUPPORTED;
    if (T < 0 || H < 1 || N < 1 || world_size < 1 || world_size > 4096 || !cu_seqlens_host || !workspace)
        return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda_kcp_workspace_bytes(T, H, K, V, N, world_size)) return KDA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return KDA_ERR_INVALID_ARG;
    const int32_t* cu = cu_seqlens_host;
    if (cu[0] != 0 || cu[N] != T) return KDA_ERR_BAD_CU_SEQLENS;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return KDA_ERR_BAD_CU_SEQLENS;

    const int W = world_size;
    const Layout L = layout(T, H, N, W);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t hs = (size_t)H * STATE_BYTES;
    const size_t fwd_bytes = kda_fwd_workspace_bytes(1, (int)(L.tmax > 0 ? L.tmax : 1), H, KD, VD, N);
    const size_t row_q = (size_t)H * KD, row_v = (size_t)H * VD;   // elements per token
    const uint16_t* q16 = static_cast<const uint16_t*>(q);
    const uint16_t* k16 = static_cast<const uint16_t*>(k);
    const uint16_t* v16 = static_cast<const uint16_t*>(v);
    uint16_t* o16 = static_cast<uint16_t*>(o);
    auto state = [&](size_t base, int i) { return reinterpret_cast<float*>(ws + base + (size_t)i * hs); };
    auto fail = [](cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; };

    // local pieces per rank
    std::vector<std::vector<Piece>> pieces(W);
    for (int r = 0; r < W; ++r) {
        const long long s0 = rank_start(T, r, W), s1 = rank_start(T, r + 1, W);
        for (int n = 0; n < N; ++n) {
            const long long a = cu[n] > s0 ? cu[n] : s0, b = cu[n + 1] < s1 ? cu[n + 1] : s1;
            if (a < b) pieces[r].push_back({n, a, b});
        }
    }
    // device cu arrays: per rank the local offsets, then [0, len] of its last piece
    std::vector<int32_t> cu_all((size_t)W * (N + 3), 0);
    for (int r = 0; r < W; ++r) {
        int32_t* c = cu_all.data() + (size_t)r * (N + 3);
        const long long s0 = rank_start(T, r, W);
        c[0] = 0;
        for (size_t i = 0; i < pieces[r].size(); ++i) c[i + 1] = (int32_t)(pieces[r][i].b - s0);
        if (!pieces[r].empty()) c[N + 2] = (int32_t)(pieces[r].back().b - pieces[r].back().a);
    }
    int32_t* cu_dev = reinterpret_cast<int32_t*>(ws + L.cu);
    kda_status st = fail(cudaMemcpyAsync(cu_dev, cu_all.data(), cu_all.size() * sizeof(int32_t),
                                         cudaMemcpyHostToDevice, stream));
    if (st != KDA_OK) return st;
    // the pageable source must outlive the copy
    if ((st = fail(cudaStreamSynchronize(stream))) != KDA_OK) return st;

    // pre-process: M_r^T and S_ext,r for every rank whose last piece continues
    std::vector<char> carries(W, 0);
    for (int r = 0; r + 1 < W; ++r) {
        if (pieces[r].empty()) continue;
        const Piece& pc = pieces[r].back();
        if (pc.b >= cu[pc.n + 1]) continue;            // the sequence ends inside rank r
        carries[r] = 1;
    }
    bool any = false;
    for (int r = 0; r < W; ++r) any = any || carries[r];
    if (any) {
        if ((st = fail(cudaMemsetAsync(ws + L.vzero, 0, (size_t)L.tmax * row_v * 2, stream))) != KDA_OK) return st;
        kda_kcp_identity_kernel<<<64, 256, 0, stream>>>(state(L.ident, 0), H);
        if ((st = fail(cudaGetLastError())) != KDA_OK) return st;
    }
    for (int r = 0; r + 1 < W; ++r) {
        if (!carries[r]) continue;
        const Piece& pc = pieces[r].back();
        const int len = (int)(pc.b - pc.a);
        const int32_t* cu1 = cu_dev + (size_t)r * (N + 3) + (N + 1);   // {0, len}
        st = kda_fwd(q16 + pc.a * row_q, k16 + pc.a * row_q, ws + L.vzero, g + pc.a * row_q, beta + pc.a * H, scale,
                     state(L.ident, 0), cu1, ws + L.scratch_o, state(L.mt, r), 1, len, H, K, V, 1, flags, ws + L.fwd,
                     fwd_bytes, stream);
        if (st != KDA_OK) return st;
        st = kda_fwd(q16 + pc.a * row_q, k16 + pc.a * row_q, v16 + pc.a * row_v, g + pc.a * row_q, beta + pc.a * H,
                     scale, nullptr, cu1, ws + L.scratch_o, state(L.ext, r), 1, len, H, K, V, 1, flags, ws + L.fwd,
                     fwd_bytes, stream);
        if (st != KDA_OK) return st;
    }

    // merge, in rank order: sin[r] is the state entering rank r (valid when
    // rank r's first piece is a continuation)
    std::vector<const float*> sin(W, nullptr);
    for (int r = 0; r + 1 < W; ++r) {
        if (pieces[r].empty()) {                       // an empty rank passes the state through
            sin[r + 1] = sin[r];
            continue;
        }
        if (!carries[r]) continue;
        const Piece& pc = pieces[r].back();
        const float* start = nullptr;
        if (pc.a > cu[pc.n]) start = sin[r];
        else if (h0 != nullptr) start = h0 + (size_t)pc.n * H * VD * KD;
        kda_kcp_merge_kernel<<<H, 256, 0, stream>>>(start, state(L.mt, r), state(L.ext, r), state(L.sin, r + 1));
        if ((st = fail(cudaGetLastError())) != KDA_OK) return st;
        sin[r + 1] = state(L.sin, r + 1);
    }

    // local forwards
    for (int n = 0; n < N; ++n)                        // empty sequences keep their initial state
        if (cu[n] == cu[n + 1] && ht != nullptr) {
            float* dst = ht + (size_t)n * H * VD * KD;
            st = h0 ? fail(cudaMemcpyAsync(dst, h0 + (size_t)n * H * VD * KD, hs, cudaMemcpyDeviceToDevice, stream))
                    : fail(cudaMemsetAsync(dst, 0, hs, stream));
            if (st != KDA_OK) return st;
        }
    for (int r = 0; r < W; ++r) {
        const std::vector<Piece>& pr = pieces[r];
        if (pr.empty()) continue;
        const long long s0 = rank_start(T, r, W), s1 = rank_start(T, r + 1, W);
        const int nl = (int)pr.size();
        for (int i = 0; i < nl; ++i) {
            float* dst = state(L.h0l, i);
            const Piece& pc = pr[i];
            if (pc.a > cu[pc.n] && sin[r] != nullptr)
                st = fail(cudaMemcpyAsync(dst, sin[r], hs, cudaMemcpyDeviceToDevice, stream));
            else if (h0 != nullptr && pc.a == cu[pc.n])
                st = fail(cudaMemcpyAsync(dst, h0 + (size_t)pc.n * H * VD * KD, hs, cudaMemcpyDeviceToDevice, stream));
            else
                st = fail(cudaMemsetAsync(dst, 0, hs, stream));
            if (st != KDA_OK) return st;
        }
        st = kda_fwd(q16 + s0 * row_q, k16 + s0 * row_q, v16 + s0 * row_v, g + s0 * row_q, beta + s0 * H, scale,
                     state(L.h0l, 0), cu_dev + (size_t)r * (N + 3), o16 + s0 * row_v, state(L.htl, 0), 1,
                     (int)(s1 - s0), H, K, V, nl, flags, ws + L.fwd, fwd_bytes, stream);
        if (st != KDA_OK) return st;
        if (ht != nullptr)
            for (int i = 0; i < nl; ++i)
                if (pr[i].b == cu[pr[i].n + 1]) {
                    st = fail(cudaMemcpyAsync(ht + (size_t)pr[i].n * H * VD * KD, state(L.htl, i), hs,
                                              cudaMemcpyDeviceToDevice, stream));
                    if (st != KDA_OK) return st;
                }
    }
    return KDA_OK;
}
