// C ABI of the KDA backward: argument checks, workspace layout and the
// launch sequence.  See include/kda.h for the contract.
#include <cmath>
#include <cstdint>

#include "../../include/kda.h"
#include "kda_bwd.cuh"
#include "kda_common.cuh"

namespace {

constexpr unsigned long long STATE_BYTES = (unsigned long long)kda::KD * kda::VD * 4ull;

long long bwd_slots(int B, int T, int N, bool varlen) {
    return varlen ? (long long)(T / kda::BT) + N + 1 : (long long)B * ((T + kda::BT - 1) / kda::BT);
}

int exact_ctas(int H, int N) {
    const long long units = (long long)N * H;
    return (int)(units < KDA_BWD_EXACT_MAX_CTAS ? units : KDA_BWD_EXACT_MAX_CTAS);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

size_t kda_bwd_workspace_bytes(int B, int T, int H, int K, int V, int N) {
    if (B < 1 || T < 0 || H < 1 || N < 1 || K != kda::KD || V != kda::VD) return 0;
    long long slots = bwd_slots(B, T, N, false);
    const long long vs = bwd_slots(B, T, N, true);
    if (vs > slots) slots = vs;
    return (size_t)(kda::WS_HEADER + (unsigned long long)slots * H * STATE_BYTES +
                    (unsigned long long)exact_ctas(H, N) * kda::BT * STATE_BYTES);
}

kda_status kda_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                   const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq, float* dk,
                   float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K, int V, int N,
                   unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (K != kda::KD || V != kda::VD) return KDA_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KDA_ERR_INVALID_ARG;
    if (B < 1 || T < 0 || H < 1 || N < 1 || H > 65535 || N > 65535) return KDA_ERR_INVALID_ARG;
    if ((flags & ~KDA_FLAG_QK_L2NORM) != 0u) return KDA_ERR_INVALID_ARG;
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

    kda::BwdParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
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
    const bool varlen = cu_seqlens != nullptr;
    const long long slots = bwd_slots(B, T, N, varlen);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.status = reinterpret_cast<uint32_t*>(ws);
    p.ckpt = reinterpret_cast<float*>(ws + kda::WS_HEADER);
    p.scratch = reinterpret_cast<float*>(ws + kda::WS_HEADER + (unsigned long long)slots * H * STATE_BYTES);
    p.scale = scale;
    p.T = T;
    p.H = H;
    p.N = N;
    p.NT = varlen ? 0 : T / kda::BT;
    p.l2norm = (flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;

    if (cudaMemsetAsync(workspace, 0, kda::WS_CLEAR, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_bwd_exact(p, nullptr, exact_ctas(H, N), stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (p.l2norm && kda::launch_l2norm_bwd(p, (long long)B * T * H, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
