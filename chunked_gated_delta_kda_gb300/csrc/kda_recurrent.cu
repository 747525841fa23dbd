// Token-by-token KDA ("fused recurrent"): the decode-phase sibling of the
// chunked forward.  Page "PyPTO-Gym chunk_kda operator: an NPU forward of
// chunked gated delta-rule linear attention", section "与其他 KDA 算子的关系"
// (relation to the other KDA operators): fused_recurrent_kda keeps an fp32
// [H, V, K] state per sequence and steps it one token at a time, with the
// state updated in place at a slot named by ssm_state_indices, speculative
// decoding through num_accepted_tokens, and the optional in-kernel q/k L2
// normalisation.  Per token (section "算子定位与算法背景"):
//   S <- diag(exp(g)) S;   S <- S + beta k (v - S^T k)^T;   o = S^T (scale q)
//
// In the page's [V, K] state layout every value row v is independent:
//   s_v <- s_v * exp(g);   s_v <- s_v + beta (v_v - k.s_v) k;   o_v = q.s_v
// so a warp owns 8 value rows, each lane 4 consecutive K entries of each
// (32 fp32 registers), and the two dot products per row are warp reductions.
// A CTA of 4 warps covers 32 value rows of one (sequence, head); the grid is
// (V / 32, H, N).  Over a sequence the token steps form one dependent chain
// per warp, so the exact recompute (long sequences) loads each token's
// inputs four tokens before its step (51 ms against 82 without the lookahead
// and 56 with eight, for the exact forward of T=65536, H=32); the decode
// kernel, one or a few tokens per sequence and bound by the state traffic,
// keeps the plain loop (the lookahead's registers cost it occupancy: 0.174
// against 0.162 ms on the decode workload).  The state is read once and written once per call (once
// per token in speculative mode), so the kernel is bound by HBM traffic on
// the state, 2 x 64 KiB per (sequence, head).
#include <cuda_bf16.h>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int REC_THREADS = 128;
constexpr int REC_ROWS = 8;                       // value rows per warp (decode)
constexpr int REC_ROWS_CTA = REC_ROWS * (REC_THREADS / 32);
// The exact recompute gives each warp two value rows when there are few
// units (with eight, 32 or fewer units put less than one warp on each SM
// sub-partition: 4.2 -> 2.9 ms for 4 units of 8192 tokens, 51 -> 49 ms for
// 32 units of 65536), eight otherwise (with two, each token's q / k / g
// rows are loaded four times as often: 6.7 -> 11.6 ms for 64 units of 8192).
constexpr int EXACT_FEW_UNITS = 32;

struct RecParams {
    const uint16_t* q;          // bf16 [B*T, H, K]
    const uint16_t* k;          // bf16 [B*T, H, K]
    const uint16_t* v;          // bf16 [B*T, H, V]
    const float* g;             // fp32 [B*T, H, K]
    const float* beta;          // fp32 [B*T, H]
    float* pool;                // fp32 [pool_slots, H, V, K], updated in place
    const int32_t* idx;         // int32 [N, stride]
    const int32_t* nacc;        // int32 [N] or null
    const int32_t* cu;          // int32 [N+1] or null
    uint16_t* o;                // bf16 [B*T, H, V]
    uint32_t* status;
    float scale;
    int T, H, N, pool_slots, stride, l2norm;
};


template <int ROWS>
__device__ __forceinline__ void store_rows(float* dst, const float (&s)[ROWS][4], int lane) {
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        *reinterpret_cast<float4*>(dst + (size_t)r * KD + 4 * lane) = make_float4(s[r][0], s[r][1], s[r][2], s[r][3]);
}

__device__ __forceinline__ void zero_output(const RecParams& p, long long bos, int len, int h, int v0, int lane) {
    if (lane != 0) return;
    for (int t = 0; t < len; ++t)
        *reinterpret_cast<uint4*>(p.o + ((size_t)(bos + t) * p.H + h) * VD + v0) = make_uint4(0, 0, 0, 0);
}

// One token's inputs as this lane loads them (raw bits; the arithmetic is
// rec_token's).  Loaded a few tokens ahead of their use, so that the
// sequential chain does not wait on global memory every token.
template <int ROWS>
struct TokIn {
    uint2 q, k;     // 4 bf16 each: K entries 4 lane .. 4 lane + 3
    float4 g;
    float beta;
    uint32_t v[ROWS / 2];   // ROWS bf16: value rows v0 .. v0 + ROWS - 1
};
constexpr int EXACT_AHEAD = 4;   // exact recompute: tokens in flight ahead of the one computed

template <int ROWS>
__device__ __forceinline__ TokIn<ROWS> load_tok(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                                                const uint16_t* __restrict__ v, const float* __restrict__ g,
                                                const float* __restrict__ beta, size_t tok, int v0, int lane) {
    TokIn<ROWS> in;
    in.q = *reinterpret_cast<const uint2*>(q + tok * KD + 4 * lane);
    in.k = *reinterpret_cast<const uint2*>(k + tok * KD + 4 * lane);
    in.g = *reinterpret_cast<const float4*>(g + tok * KD + 4 * lane);
    in.beta = beta[tok];
    if constexpr (ROWS == 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(v + tok * VD + v0);
        in.v[0] = u.x; in.v[1] = u.y; in.v[2] = u.z; in.v[3] = u.w;
    } else {
        static_assert(ROWS == 2, "two or eight value rows per warp");
        in.v[0] = *reinterpret_cast<const uint32_t*>(v + tok * VD + v0);
    }
    return in;
}

// All-reduce two per-lane partial sums over the warp: one exchange on lane
// bit 4 leaves each half-warp with one row's pair sums, a butterfly over the
// other four bits completes it, then both totals are fetched.
__device__ __forceinline__ void warp_sum2(float (&a)[2], int lane) {
    const bool h16 = lane & 16;
    float b = (h16 ? a[1] : a[0]) + __shfl_xor_sync(0xffffffffu, h16 ? a[0] : a[1], 16);
#pragma unroll
    for (int m = 8; m > 0; m >>= 1) b += __shfl_xor_sync(0xffffffffu, b, m);
    a[0] = __shfl_sync(0xffffffffu, b, 0);
    a[1] = __shfl_sync(0xffffffffu, b, 16);
}

// One token of the recurrence on this warp's ROWS value rows (row v0 + r in
// s[r], lane owning K entries 4 lane .. 4 lane + 3): decay, delta update,
// read-out; lane 0 writes the ROWS bf16 outputs.  `tok` indexes (token, head).
template <int ROWS>
__device__ __forceinline__ void rec_token(const TokIn<ROWS>& in, uint16_t* __restrict__ o, float scale, bool l2norm,
                                          size_t tok, int v0, int lane, float (&s)[ROWS][4]) {
    float qv[4], kv[4];
    qv[0] = __uint_as_float(in.q.x << 16); qv[1] = __uint_as_float(in.q.x & 0xffff0000u);
    qv[2] = __uint_as_float(in.q.y << 16); qv[3] = __uint_as_float(in.q.y & 0xffff0000u);
    kv[0] = __uint_as_float(in.k.x << 16); kv[1] = __uint_as_float(in.k.x & 0xffff0000u);
    kv[2] = __uint_as_float(in.k.y << 16); kv[3] = __uint_as_float(in.k.y & 0xffff0000u);
    const float4 gv = in.g;
    const float bt = in.beta;
    float vv[ROWS];
#pragma unroll
    for (int j = 0; j < ROWS / 2; ++j) {
        vv[2 * j] = __uint_as_float(in.v[j] << 16);
        vv[2 * j + 1] = __uint_as_float(in.v[j] & 0xffff0000u);
    }

    float qs = scale, ks = 1.f;
    if (l2norm) {   // x / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
        const float sq = warp_sum(qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3]);
        const float sk = warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]);
        qs *= rsqrtf(sq + 1e-6f);
        ks = rsqrtf(sk + 1e-6f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        qv[i] *= qs;
        kv[i] *= ks;
    }
    const float e[4] = {__expf(gv.x), __expf(gv.y), __expf(gv.z), __expf(gv.w)};

    auto reduce = [&](float (&d)[ROWS]) {
        if constexpr (ROWS == 8) warp_sum8(d, lane);
        else warp_sum2(d, lane);
    };
    // decay, then k . s_v
    float dot[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[r][i] *= e[i];
            acc = fmaf(kv[i], s[r][i], acc);
        }
        dot[r] = acc;
    }
    reduce(dot);
    // delta update, then q . s_v
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const float delta = bt * (vv[r] - dot[r]);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[r][i] = fmaf(kv[i], delta, s[r][i]);
            acc = fmaf(qv[i], s[r][i], acc);
        }
        dot[r] = acc;
    }
    reduce(dot);
    if (lane == 0) {
        __nv_bfloat162 o2[ROWS / 2];
#pragma unroll
        for (int j = 0; j < ROWS / 2; ++j) o2[j] = __floats2bfloat162_rn(dot[2 * j], dot[2 * j + 1]);
        if constexpr (ROWS == 8) *reinterpret_cast<uint4*>(o + tok * VD + v0) = *reinterpret_cast<const uint4*>(o2);
        else *reinterpret_cast<__nv_bfloat162*>(o + tok * VD + v0) = o2[0];
    }
}

// The same token step for two value rows with one warp reduction instead of
// two: with s_d the decayed state and delta = beta (v - k.s_d), the read-out
// of the updated state is q.s_d + delta (q.k), so k.s_d, q.s_d (both rows)
// and q.k are reduced together.  The exact recompute's chain per token is
// then one reduction long.
__device__ __forceinline__ void rec_token_one_reduction(const TokIn<2>& in, uint16_t* __restrict__ o, float scale,
                                                        bool l2norm, size_t tok, int v0, int lane, float (&s)[2][4]) {
    float qv[4], kv[4];
    qv[0] = __uint_as_float(in.q.x << 16); qv[1] = __uint_as_float(in.q.x & 0xffff0000u);
    qv[2] = __uint_as_float(in.q.y << 16); qv[3] = __uint_as_float(in.q.y & 0xffff0000u);
    kv[0] = __uint_as_float(in.k.x << 16); kv[1] = __uint_as_float(in.k.x & 0xffff0000u);
    kv[2] = __uint_as_float(in.k.y << 16); kv[3] = __uint_as_float(in.k.y & 0xffff0000u);
    const float vv[2] = {__uint_as_float(in.v[0] << 16), __uint_as_float(in.v[0] & 0xffff0000u)};
    float qs = scale, ks = 1.f;
    if (l2norm) {   // x / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
        const float sq = warp_sum(qv[0] * qv[0] + qv[1] * qv[1] + qv[2] * qv[2] + qv[3] * qv[3]);
        const float sk = warp_sum(kv[0] * kv[0] + kv[1] * kv[1] + kv[2] * kv[2] + kv[3] * kv[3]);
        qs *= rsqrtf(sq + 1e-6f);
        ks = rsqrtf(sk + 1e-6f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        qv[i] *= qs;
        kv[i] *= ks;
    }
    const float e[4] = {__expf(in.g.x), __expf(in.g.y), __expf(in.g.z), __expf(in.g.w)};
    // [k.s_d row 0, row 1, q.s_d row 0, row 1, q.k, -, -, -]
    float d[8];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float ak = 0.f, aq = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[r][i] *= e[i];
            ak = fmaf(kv[i], s[r][i], ak);
            aq = fmaf(qv[i], s[r][i], aq);
        }
        d[r] = ak;
        d[2 + r] = aq;
    }
    d[4] = qv[0] * kv[0] + qv[1] * kv[1] + qv[2] * kv[2] + qv[3] * kv[3];
    d[5] = d[6] = d[7] = 0.f;
    warp_sum8(d, lane);
    float out[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float delta = in.beta * (vv[r] - d[r]);
#pragma unroll
        for (int i = 0; i < 4; ++i) s[r][i] = fmaf(kv[i], delta, s[r][i]);
        out[r] = fmaf(delta, d[4], d[2 + r]);
    }
    if (lane == 0)
        *reinterpret_cast<__nv_bfloat162*>(o + tok * VD + v0) = __floats2bfloat162_rn(out[0], out[1]);
}

// Tokens 0 .. len - 1 of one (sequence, head) starting at packed token bos:
// AHEAD = 0 loads each token's inputs right before its step; otherwise a
// ring of AHEAD loaded inputs (slot i holds token t0 + i of the current
// group), each refilled with the token AHEAD on as soon as it is consumed.
// after(t) runs after token t's update.
template <int ROWS, int AHEAD, class After>
__device__ __forceinline__ void rec_tokens(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                                           const uint16_t* __restrict__ v, const float* __restrict__ g,
                                           const float* __restrict__ beta, uint16_t* __restrict__ o, float scale,
                                           bool l2norm, long long bos, int len, int H, int h, int v0, int lane,
                                           float (&s)[ROWS][4], After after) {
    if constexpr (AHEAD == 0) {
        for (int t = 0; t < len; ++t) {
            const size_t tok = (size_t)(bos + t) * H + h;
            rec_token<ROWS>(load_tok<ROWS>(q, k, v, g, beta, tok, v0, lane), o, scale, l2norm, tok, v0, lane, s);
            after(t);
        }
    } else {
        TokIn<ROWS> ring[AHEAD];
#pragma unroll
        for (int i = 0; i < AHEAD; ++i)
            if (i < len) ring[i] = load_tok<ROWS>(q, k, v, g, beta, (size_t)(bos + i) * H + h, v0, lane);
        for (int t0 = 0; t0 < len; t0 += AHEAD) {
#pragma unroll
            for (int i = 0; i < AHEAD; ++i) {
                const int t = t0 + i;
                if (t < len) {
                    const TokIn<ROWS> cur = ring[i];
                    if (t + AHEAD < len)
                        ring[i] = load_tok<ROWS>(q, k, v, g, beta, (size_t)(bos + t + AHEAD) * H + h, v0, lane);
                    if constexpr (ROWS == 2)
                        rec_token_one_reduction(cur, o, scale, l2norm, (size_t)(bos + t) * H + h, v0, lane, s);
                    else
                        rec_token<ROWS>(cur, o, scale, l2norm, (size_t)(bos + t) * H + h, v0, lane, s);
                    after(t);
                }
            }
        }
    }
}

}  // namespace

__global__ void __launch_bounds__(REC_THREADS) kda_recurrent_kernel(const RecParams p) {
    const int h = (int)blockIdx.y, n = (int)blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v0 = (int)blockIdx.x * REC_ROWS_CTA + warp * REC_ROWS;
    const int H = p.H;
    const bool first = blockIdx.x == 0 && threadIdx.x == 0;   // reports errors once per (n, h)

    // sequence bounds (section "主机侧 wrapper 与输入校验": fixed length is N = B
    // sequences of T tokens; varlen offsets come from cu_seqlens on the device)
    long long bos;
    int len;
    if (p.cu == nullptr) {
        bos = (long long)n * p.T;
        len = p.T;
    } else {
        const int a = p.cu[n], b = p.cu[n + 1];
        if (a < 0 || b < a || b > p.T || (n == 0 && a != 0) || (n == p.N - 1 && b != p.T)) {
            if (first && h == 0) atomicOr(p.status, STATUS_BAD_CU);
            return;
        }
        bos = a;
        len = b - a;
    }
    if (len == 0) return;

    // state slots: read slot, and (speculative mode) one write slot per token
    const int32_t* row = p.idx + (size_t)n * p.stride;
    int rslot;
    if (p.nacc == nullptr) {
        rslot = row[0];
    } else {
        const int acc = p.nacc[n];
        bool ok = acc >= 1 && acc <= p.stride && len <= p.stride;
        if (ok) {
            for (int t = 0; t < len; ++t) ok = ok && row[t] < p.pool_slots;
        }
        if (!ok) {
            if (first && h == 0) atomicOr(p.status, STATUS_BAD_INDEX);
            zero_output(p, bos, len, h, v0, lane);
            return;
        }
        rslot = row[acc - 1];
    }
    if (rslot >= p.pool_slots) {
        if (first && h == 0) atomicOr(p.status, STATUS_BAD_INDEX);
        zero_output(p, bos, len, h, v0, lane);
        return;
    }
    if (rslot < 0) {   // padding entry: no state, no output
        zero_output(p, bos, len, h, v0, lane);
        return;
    }

    float s[REC_ROWS][4];
    {
        const float* src = p.pool + (((size_t)rslot * H + h) * VD + v0) * KD;
#pragma unroll
        for (int r = 0; r < REC_ROWS; ++r) {
            const float4 x = *reinterpret_cast<const float4*>(src + (size_t)r * KD + 4 * lane);
            s[r][0] = x.x; s[r][1] = x.y; s[r][2] = x.z; s[r][3] = x.w;
        }
    }

    rec_tokens<REC_ROWS, 0>(p.q, p.k, p.v, p.g, p.beta, p.o, p.scale, p.l2norm != 0, bos, len, H, h, v0, lane, s, [&](int t) {
        if (p.nacc != nullptr) {   // speculative mode: the state after token t goes to slot row[t]
            const int ws = row[t];
            if (ws >= 0) store_rows(p.pool + (((size_t)ws * H + h) * VD + v0) * KD, s, lane);
        }
    });
    if (p.nacc == nullptr) store_rows(p.pool + (((size_t)rslot * H + h) * VD + v0) * KD, s, lane);
}

// Exact recomputation for the chunked forward (one (sequence, head) per
// blockIdx.y/z, 8 or 32 value rows per CTA): the (sequence, head) units in which
// some chunk's in-chunk decay exceeded the range of exact factored products
// (flagged by the chunk-parallel kernel) are recomputed here token by token,
// from h0, overwriting the chunked result's o and final state.  The
// recurrence is the same per-token rule, so it is exact for any decay.
template <int ROWS>
__global__ void __launch_bounds__(REC_THREADS) kda_exact_kernel(const FwdParams p, const uint32_t* flags,
                                                                int l2norm) {
    const int h = (int)blockIdx.y, n = (int)blockIdx.z;
    const int H = p.H;
    if (flags[(size_t)n * H + h] == 0u) return;   // uniform
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v0 = (int)blockIdx.x * ROWS * (REC_THREADS / 32) + warp * ROWS;
    long long bos;
    int len;
    if (!seq_bounds(p, n, bos, len)) return;
    const size_t st = (((size_t)n * H + h) * VD + v0) * KD;
    float s[ROWS][4];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.h0 != nullptr) x = *reinterpret_cast<const float4*>(p.h0 + st + (size_t)r * KD + 4 * lane);
        s[r][0] = x.x; s[r][1] = x.y; s[r][2] = x.z; s[r][3] = x.w;
    }
    rec_tokens<ROWS, EXACT_AHEAD>(p.q, p.k, p.v, p.g, p.beta, p.o, p.scale, l2norm != 0, bos, len, H, h, v0, lane, s,
                                  [](int) {});
    if (p.ht != nullptr) store_rows(p.ht + st, s, lane);
}

cudaError_t launch_exact(const FwdParams& p, const uint32_t* flags, bool l2norm, cudaStream_t stream) {
    if (p.N == 0) return cudaSuccess;
    if ((long long)p.N * p.H <= EXACT_FEW_UNITS) {
        const dim3 grid((unsigned)(VD / (2 * (REC_THREADS / 32))), (unsigned)p.H, (unsigned)p.N);
        kda_exact_kernel<2><<<grid, REC_THREADS, 0, stream>>>(p, flags, l2norm ? 1 : 0);
    } else {
        const dim3 grid((unsigned)(VD / REC_ROWS_CTA), (unsigned)p.H, (unsigned)p.N);
        kda_exact_kernel<REC_ROWS><<<grid, REC_THREADS, 0, stream>>>(p, flags, l2norm ? 1 : 0);
    }
    return cudaGetLastError();
}

}  // namespace kda

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" kda_status kda_fused_recurrent(const void* q, const void* k, const void* v, const float* g,
                                          const float* beta, float scale, float* state_pool, int pool_slots,
                                          const int32_t* ssm_state_indices, int indices_stride,
                                          const int32_t* num_accepted_tokens, const int32_t* cu_seqlens,
                                          void* o, int B, int T, int H, int K, int V, int N, unsigned flags,
                                          void* workspace, cudaStream_t stream) {
    using namespace kda;
    if (K != KD || V != VD) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || N < 0 || pool_slots <= 0 || indices_stride <= 0) return KDA_ERR_INVALID_ARG;
    if ((flags & ~KDA_FLAG_QK_L2NORM) != 0u) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr) {
        if (N != B) return KDA_ERR_INVALID_ARG;
    } else if (B != 1) {
        return KDA_ERR_INVALID_ARG;
    }
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0u) return KDA_ERR_INVALID_ARG;
    if (state_pool == nullptr || ssm_state_indices == nullptr) return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(state_pool) & 15u) != 0u) return KDA_ERR_INVALID_ARG;
    const bool any_tokens = (long long)B * T > 0;
    if (any_tokens) {
        const void* ptrs[] = {q, k, v, g, o};
        for (const void* ptr : ptrs)
            if (ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0u) return KDA_ERR_INVALID_ARG;
        if (beta == nullptr || (reinterpret_cast<uintptr_t>(beta) & 3u) != 0u) return KDA_ERR_INVALID_ARG;
    }
    if (cudaMemsetAsync(workspace, 0, WS_CLEAR, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (!any_tokens || N == 0) return KDA_OK;

    RecParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.g = g;
    p.beta = beta;
    p.pool = state_pool;
    p.idx = ssm_state_indices;
    p.nacc = num_accepted_tokens;
    p.cu = cu_seqlens;
    p.o = static_cast<uint16_t*>(o);
    p.status = static_cast<uint32_t*>(workspace);
    p.scale = (scale > 0.f) ? scale : 0.08838834764831845f;   // 128^-0.5
    p.T = cu_seqlens == nullptr ? T : B * T;
    p.H = H;
    p.N = N;
    p.pool_slots = pool_slots;
    p.stride = indices_stride;
    p.l2norm = (flags & KDA_FLAG_QK_L2NORM) ? 1 : 0;
    const dim3 grid((unsigned)(VD / REC_ROWS_CTA), (unsigned)H, (unsigned)N);
    kda_recurrent_kernel<<<grid, REC_THREADS, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
