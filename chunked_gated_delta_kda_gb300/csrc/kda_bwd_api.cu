// C ABI of the KDA backward: argument checks, workspace layout and the
// launch sequence.  See include/kda.h for the contract.
//
// Chunked path (default), on the caller's stream:
//   1. the forward's chunk-parallel kernel (transition tiles, exact flags);
//   2. the forward's scan in state-only mode, storing S entering each chunk;
//   3. kda_bwd_tiles_kernel: Nm^T, Qe^T do, Dg at mirrored chunk positions;
//   4. the scan again on those tiles from dht: dS at every chunk end, dh0;
//   5. kda_bwd_tc_kernel: the per-chunk chain rule in chunked form on the
//      tensor cores; kda_bwd_chunk_kernel (per-token fp32 replay) takes the
//      chunks whose decay leaves its range (or every chunk, with
//      KDA_FLAG_BWD_CHUNK_FP32);
//   6. the token-by-token backward for the (sequence, head) units the
//      forward flagged as beyond its factoring range;
//   7. the q/k normalisation chain rule when requested.
// KDA_FLAG_BWD_TOKEN_EXACT runs the token-by-token backward for every unit.
#include <cmath>
#include <cstdint>

#include "../../include/kda.h"
#include "kda_bwd.cuh"
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_prep(const FwdParams& p, bool l2norm, cudaStream_t stream);
cudaError_t launch_scan(const FwdParams& p, cudaStream_t stream);
uint32_t debug_wait_limit();
}  // namespace kda

namespace {

constexpr unsigned long long STATE_BYTES = (unsigned long long)kda::KD * kda::VD * 4ull;

long long bwd_slots(int B, int T, int N, bool varlen) {
    return varlen ? (long long)(T / kda::BT) + N + 1 : (long long)B * ((T + kda::BT - 1) / kda::BT);
}

long long max_slots(int B, int T, int N) {
    const long long a = bwd_slots(B, T, N, false), b = bwd_slots(B, T, N, true);
    return a > b ? a : b;
}

unsigned long long r256(unsigned long long x) { return (x + 255ull) / 256ull * 256ull; }

// Scratch buffers (one per resident CTA of the per-chunk and token-by-token kernels).
int scratch_ctas(long long items, int H, int N) {
    long long u = items > (long long)N * H ? items : (long long)N * H;
    return (int)(u < KDA_BWD_EXACT_MAX_CTAS ? u : KDA_BWD_EXACT_MAX_CTAS);
}

struct Layout {
    unsigned long long tiles, flags, btiles, ckpt_s, ckpt_d, ckpt_x, skip, scratch, total;
};

Layout layout(int B, int T, int H, int N) {
    const unsigned long long items = (unsigned long long)max_slots(B, T, N) * (unsigned long long)H;
    Layout L;
    L.tiles = kda::ws_tiles_offset(items);
    L.flags = L.tiles + items * kda::TILE_BYTES;
    L.btiles = L.flags + r256((unsigned long long)N * H * 4ull);
    L.ckpt_s = L.btiles + items * kda::TILE_BYTES;
    L.ckpt_d = L.ckpt_s + items * STATE_BYTES;
    L.ckpt_x = L.ckpt_d + items * STATE_BYTES;
    L.skip = L.ckpt_x + items * STATE_BYTES;
    L.scratch = L.skip + r256(items * 4ull);
    L.total = L.scratch + (unsigned long long)scratch_ctas((long long)items, H, N) * kda::BT * STATE_BYTES;
    return L;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace kda {
// Byte offset of the chunk states in kda_bwd's workspace (kda_fwd stores them
// there under KDA_FLAG_SAVE_FOR_BWD).
unsigned long long bwd_chunk_state_offset(int B, int T, int H, int N) { return layout(B, T, H, N).ckpt_s; }
}  // namespace kda

extern "C" {

size_t kda_bwd_workspace_bytes(int B, int T, int H, int K, int V, int N) {
    if (B < 1 || T < 0 || H < 1 || N < 1 || K != kda::KD || V != kda::VD) return 0;
    return (size_t)layout(B, T, H, N).total;
}

static kda_status bwd_impl(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                           const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq,
                           float* dk, float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K,
                           int V, int N, unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           cudaEvent_t* ev) {
    if (K != kda::KD || V != kda::VD) return KDA_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KDA_ERR_INVALID_ARG;
    if (B < 1 || T < 0 || H < 1 || N < 1 || H > 65535 || N > 65535) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(KDA_FLAG_QK_L2NORM | KDA_FLAG_BWD_TOKEN_EXACT | KDA_FLAG_BWD_CHUNK_FP32 |
                   KDA_FLAG_BWD_REUSE_FWD | KDA_FLAG_BWD_UMMA)) != 0u)
        return KDA_ERR_INVALID_ARG;
    const bool reuse = (flags & KDA_FLAG_BWD_REUSE_FWD) != 0u;
    if (reuse && (flags & KDA_FLAG_BWD_TOKEN_EXACT)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr) {
        if (N != B || T % kda::BT != 0) return KDA_ERR_INVALID_ARG;
    } else if (B != 1) {
        return KDA_ERR_INVALID_ARG;
    }
    if (T > 0) {
        const void* ptrs[] = {q, k, v, g, dout, dq, dk, dv, dg};
        for (const void* ptr : ptrs)
            if (ptr == nullptr || !a16(ptr)) return KDA_ERR_INVALID_ARG;
        if (!beta || !dbeta || (reinterpret_cast<uintptr_t>(beta) & 3u) || (reinterpret_cast<uintptr_t>(dbeta) & 3u))
            return KDA_ERR_INVALID_ARG;
    }
    if ((h0 && !a16(h0)) || (dht && !a16(dht)) || (dh0 && !a16(dh0))) return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda_bwd_workspace_bytes(B, T, H, K, V, N)) return KDA_ERR_INVALID_ARG;
    if ((long long)B * T * H * kda::KD >= (1ll << 62)) return KDA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || std::isnan(scale)) scale = 1.0f / std::sqrt((float)K);

    const bool varlen = cu_seqlens != nullptr;
    const bool l2norm = (flags & KDA_FLAG_QK_L2NORM) != 0u;
    const unsigned long long items = (unsigned long long)max_slots(B, T, N) * (unsigned long long)H;
    const Layout L = layout(B, T, H, N);
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    kda::FwdParams fp{};
    fp.q = static_cast<const uint16_t*>(q);
    fp.k = static_cast<const uint16_t*>(k);
    fp.v = static_cast<const uint16_t*>(v);
    fp.g = g;
    fp.beta = beta;
    fp.h0 = h0;
    fp.cu = cu_seqlens;
    fp.o = nullptr;
    fp.ht = nullptr;
    fp.status = reinterpret_cast<uint32_t*>(ws);
    fp.wide_count = reinterpret_cast<uint32_t*>(ws) + 1;
    fp.wide_list = reinterpret_cast<int32_t*>(ws + kda::WS_HEADER);
    fp.tiles = ws + L.tiles;
    fp.exact_flags = reinterpret_cast<uint32_t*>(ws + L.flags);
    fp.ckpt = reinterpret_cast<float*>(ws + L.ckpt_s);
    fp.scale = scale;
    fp.wait_limit = kda::debug_wait_limit();
    fp.T = T;
    fp.H = H;
    fp.N = N;
    fp.NT = varlen ? 0 : T / kda::BT;
    fp.nslots = varlen ? T / kda::BT + N + 1 : N * (T / kda::BT);

    kda::BwdParams p{};
    p.q = fp.q;
    p.k = fp.k;
    p.v = fp.v;
    p.g = g;
    p.beta = beta;
    p.h0 = h0;
    p.cu = cu_seqlens;
    p.dout = static_cast<const uint16_t*>(dout);
    p.dht = dht;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dg = dg;
    p.dbeta = dbeta;
    p.dh0 = dh0;
    p.ckpt = reinterpret_cast<float*>(ws + L.ckpt_x);
    p.scratch = reinterpret_cast<float*>(ws + L.scratch);
    p.ckpt_s = reinterpret_cast<const float*>(ws + L.ckpt_s);
    p.ckpt_d = reinterpret_cast<const float*>(ws + L.ckpt_d);
    p.tc_skip = nullptr;
    p.status = fp.status;
    p.scale = scale;
    p.T = T;
    p.H = H;
    p.N = N;
    p.NT = fp.NT;
    p.l2norm = l2norm ? 1 : 0;
    const int ctas = scratch_ctas((long long)items, H, N);

    auto mark = [&](int i) { return ev == nullptr || cudaEventRecord(ev[i], stream) == cudaSuccess; };
    if (cudaMemsetAsync(workspace, 0, kda::WS_CLEAR, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (!mark(0)) return KDA_ERR_CUDA;
    if (flags & KDA_FLAG_BWD_TOKEN_EXACT) {
        if (kda::launch_bwd_exact(p, nullptr, ctas < N * H ? ctas : N * H, stream) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        if (!reuse) {   // else: the tiles, flags and chunk states of the saving forward are in place
            if (cudaMemsetAsync(fp.exact_flags, 0, (size_t)N * H * 4, stream) != cudaSuccess) return KDA_ERR_CUDA;
            if (fp.nslots > 0 && kda::launch_prep(fp, l2norm, stream) != cudaSuccess) return KDA_ERR_CUDA;
            if (kda::launch_scan(fp, stream) != cudaSuccess) return KDA_ERR_CUDA;
        }
        if (!mark(1)) return KDA_ERR_CUDA;
        if (kda::launch_bwd_tiles(fp, ws + L.btiles, p.dout, stream) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark(2)) return KDA_ERR_CUDA;
        kda::FwdParams rp = fp;   // the reverse state pass
        rp.tiles = ws + L.btiles;
        rp.h0 = dht;
        rp.ht = dh0;
        rp.ckpt = reinterpret_cast<float*>(ws + L.ckpt_d);
        if (kda::launch_scan(rp, stream) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark(3)) return KDA_ERR_CUDA;
        if (flags & KDA_FLAG_BWD_CHUNK_FP32) {
            if (kda::launch_bwd_chunk(p, fp, ctas, stream) != cudaSuccess) return KDA_ERR_CUDA;
        } else {
            // tensor-core chunks first; the per-token kernel takes the chunks it left
            kda::BwdParams tp = p;
            tp.tc_skip = reinterpret_cast<uint32_t*>(ws + L.skip);
            if (cudaMemsetAsync(tp.tc_skip, 0, (size_t)items * 4, stream) != cudaSuccess) return KDA_ERR_CUDA;
            const cudaError_t e = (flags & KDA_FLAG_BWD_UMMA) ? kda::launch_bwd_umma(tp, fp, ctas, stream)
                                                               : kda::launch_bwd_tc(tp, fp, ctas, stream);
            if (e != cudaSuccess) return KDA_ERR_CUDA;
            if (kda::launch_bwd_chunk(tp, fp, ctas, stream) != cudaSuccess) return KDA_ERR_CUDA;
        }
        if (!mark(4)) return KDA_ERR_CUDA;
        if (kda::launch_bwd_exact(p, fp.exact_flags, ctas < N * H ? ctas : N * H, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    if (l2norm && kda::launch_l2norm_bwd(p, (long long)B * T * H, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (!mark(5)) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                   const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq, float* dk,
                   float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K, int V, int N,
                   unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return bwd_impl(q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, B, T, H, K, V, N,
                    flags, workspace, workspace_bytes, stream, nullptr);
}

kda_status kda_bwd_timed(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                         const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq,
                         float* dk, float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K, int V,
                         int N, unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         cudaEvent_t* stage_events) {
    if (!stage_events) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!stage_events[i]) return KDA_ERR_INVALID_ARG;
    if (flags & KDA_FLAG_BWD_TOKEN_EXACT) return KDA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht, dq, dk, dv, dg, dbeta, dh0, B, T, H, K, V, N,
                    flags, workspace, workspace_bytes, stream, stage_events);
}

}  // extern "C"
