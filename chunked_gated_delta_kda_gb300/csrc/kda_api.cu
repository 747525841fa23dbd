// C ABI of the chunked KDA forward: host-side argument checks, workspace
// sizing and the launch sequence (status reset, prep, scan) on the caller's
// stream.  See include/kda.h for the contract.
#include <cmath>
#include <cstdint>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace kda {
// Test hooks (kda_debug_set): poll limit of the bounded waits (0: the
// kernels' default) and one-shot debug bits for the next forward.
static uint32_t g_wait_limit = 0;
static uint32_t g_debug_once = 0;
uint32_t debug_wait_limit() { return g_wait_limit; }
unsigned long long bwd_chunk_state_offset(int B, int T, int H, int N);
cudaError_t launch_prep(const FwdParams& p, bool l2norm, cudaStream_t stream);
cudaError_t launch_scan(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_exact(const FwdParams& p, const uint32_t* flags, bool l2norm, cudaStream_t stream);
}  // namespace kda

namespace {

// Upper bound on chunk slots: fixed length uses B * T/128, varlen at most
// floor(T/128) + N + 1 (see kda_common.cuh).
long long max_slots(int B, int T, int N) {
    const long long fixed = (long long)B * ((T + kda::BT - 1) / kda::BT);
    const long long varlen = (long long)(T / kda::BT) + N + 1;
    return fixed > varlen ? fixed : varlen;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

// Bytes of the per-(sequence, head) exact-recompute flags after the tiles.
static unsigned long long flags_bytes(int H, int N) {
    return (((unsigned long long)N * (unsigned long long)H * 4ull + 255ull) / 256ull) * 256ull;
}

size_t kda_fwd_workspace_bytes(int B, int T, int H, int K, int V, int N) {
    if (B < 1 || T < 0 || H < 1 || N < 1 || K != kda::KD || V != kda::VD) return 0;
    const unsigned long long items = (unsigned long long)max_slots(B, T, N) * (unsigned long long)H;
    return (size_t)(kda::ws_tiles_offset(items) + items * kda::TILE_BYTES + flags_bytes(H, N));
}

static kda_status fwd_impl(const void* q, const void* k, const void* v, const float* g, const float* beta,
                           float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht, int B, int T,
                           int H, int K, int V, int N, unsigned flags, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream, cudaEvent_t* ev) {
    if (K != kda::KD || V != kda::VD) return KDA_ERR_UNSUPPORTED;
    // With T == 0 there is nothing to read or write (frameworks hand out null
    // pointers for empty tensors); only the state tensors and workspace are used.
    if (!workspace) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (B < 1 || T < 0 || H < 1 || N < 1 || H > 65535 || N > 65535) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(KDA_FLAG_QK_L2NORM | KDA_FLAG_SAVE_FOR_BWD | KDA_FLAG_FWD_TOKEN_EXACT)) != 0u)
        return KDA_ERR_INVALID_ARG;
    const bool save = (flags & KDA_FLAG_SAVE_FOR_BWD) != 0u;
    const bool token_exact = (flags & KDA_FLAG_FWD_TOKEN_EXACT) != 0u;
    if (save && token_exact) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr) {
        if (N != B || T % kda::BT != 0) return KDA_ERR_INVALID_ARG;
    } else {
        if (B != 1) return KDA_ERR_INVALID_ARG;
    }
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || (reinterpret_cast<uintptr_t>(beta) & 3u) ||
        !aligned16(o) ||
        (h0 && !aligned16(h0)) || (ht && !aligned16(ht)) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < kda_fwd_workspace_bytes(B, T, H, K, V, N)) return KDA_ERR_INVALID_ARG;
    if (save && workspace_bytes < kda_bwd_workspace_bytes(B, T, H, K, V, N)) return KDA_ERR_INVALID_ARG;
    const long long total_rows = (long long)B * T * H;
    if (total_rows * kda::KD >= (1ll << 62)) return KDA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || std::isnan(scale)) scale = 1.0f / std::sqrt((float)K);

    kda::FwdParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.g = g;
    p.beta = beta;
    p.h0 = h0;
    p.cu = cu_seqlens;
    p.o = static_cast<uint16_t*>(o);
    p.ht = ht;
    const unsigned long long items = (unsigned long long)max_slots(B, T, N) * (unsigned long long)H;
    p.status = static_cast<uint32_t*>(workspace);
    p.wide_count = static_cast<uint32_t*>(workspace) + 1;
    p.wide_list = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + kda::WS_HEADER);
    p.tiles = static_cast<uint8_t*>(workspace) + kda::ws_tiles_offset(items);
    p.exact_flags =
        reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + kda::ws_tiles_offset(items) + items * kda::TILE_BYTES);
    // with KDA_FLAG_SAVE_FOR_BWD the scan also stores the state entering every
    // chunk where kda_bwd's workspace layout keeps it (the tiles and flags are
    // already where kda_bwd reads them: its layout starts with this one)
    p.ckpt = save ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kda::bwd_chunk_state_offset(B, T, H, N))
                  : nullptr;
    p.scale = scale;
    p.T = T;
    p.H = H;
    p.N = N;
    p.wait_limit = kda::g_wait_limit;
    p.debug = kda::g_debug_once;
    kda::g_debug_once = 0;
    if (cu_seqlens == nullptr) {
        p.NT = T / kda::BT;
        p.nslots = N * p.NT;
    } else {
        p.NT = 0;
        p.nslots = T / kda::BT + N + 1;
    }

    if (cudaMemsetAsync(workspace, 0, kda::WS_CLEAR, stream) != cudaSuccess) return KDA_ERR_CUDA;
    // token-exact: every unit flagged (non-zero words), nothing chunked runs
    if (cudaMemsetAsync(p.exact_flags, token_exact ? 1 : 0, (size_t)N * H * 4, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (token_exact) {
        if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return KDA_ERR_CUDA;
        if (kda::launch_exact(p, p.exact_flags, (flags & KDA_FLAG_QK_L2NORM) != 0u, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return KDA_ERR_CUDA;
        return KDA_OK;
    }
    if (p.nslots > 0) {
        if (kda::launch_prep(p, (flags & KDA_FLAG_QK_L2NORM) != 0u, stream) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_scan(p, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_exact(p, p.exact_flags, (flags & KDA_FLAG_QK_L2NORM) != 0u, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                   const float* h0, const int32_t* cu_seqlens, void* o, float* ht, int B, int T, int H, int K, int V,
                   int N, unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return fwd_impl(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, B, T, H, K, V, N, flags, workspace,
                    workspace_bytes, stream, nullptr);
}

kda_status kda_fwd_timed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht, int B, int T,
                         int H, int K, int V, int N, unsigned flags, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream, cudaEvent_t* stage_events) {
    if (!stage_events || !stage_events[0] || !stage_events[1] || !stage_events[2]) return KDA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, B, T, H, K, V, N, flags, workspace,
                    workspace_bytes, stream, stage_events);
}

kda_status kda_get_status(const void* workspace, cudaStream_t stream) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kda::STATUS_BAD_CU) return KDA_ERR_BAD_CU_SEQLENS;
    if (word & kda::STATUS_TIMEOUT) return KDA_ERR_TIMEOUT;
    if (word & kda::STATUS_BAD_INDEX) return KDA_ERR_BAD_STATE_INDEX;
    return KDA_OK;
}

kda_status kda_debug_set(int what, unsigned value) {
    switch (what) {
        case KDA_DEBUG_WAIT_LIMIT: kda::g_wait_limit = value; return KDA_OK;
        case KDA_DEBUG_DROP_SCAN_LOAD:
            kda::g_debug_once = value ? (kda::g_debug_once | kda::DEBUG_DROP_SCAN_LOAD)
                                      : (kda::g_debug_once & ~kda::DEBUG_DROP_SCAN_LOAD);
            return KDA_OK;
    }
    return KDA_ERR_INVALID_ARG;
}

const char* kda_status_str(kda_status status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument (pointer, size, alignment or packing)";
        case KDA_ERR_UNSUPPORTED: return "unsupported head size (K and V must be 128)";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_BAD_CU_SEQLENS: return "device found cu_seqlens invalid";
        case KDA_ERR_TIMEOUT: return "a bounded device wait ran out";
        case KDA_ERR_TOO_LARGE: return "problem too large for the static no-alloc scratch";
        case KDA_ERR_BAD_STATE_INDEX: return "device found a state slot index or accepted-token count out of range";
    }
    return "unknown status";
}

}  // extern "C"
