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
// inputs ahead of its step, four tokens ahead with eight rows per warp and
// one four-token window ahead with two (51 ms against 82 without the
// lookahead and 56 with eight, for the exact forward of T=65536, H=32); the
// decode kernel, one or a few tokens per sequence and bound by the state
// traffic, keeps the plain loop (the lookahead's registers cost it
// occupancy: 0.174 against 0.162 ms on the decode workload).  The state is
// read once and written once per call (once per token in speculative mode),
// so the kernel is bound by HBM traffic on the state, 2 x 64 KiB per
// (sequence, head).
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
// 32 units of 65536), stepped four tokens at a time with one warp reduction
// per window (2.9 -> 2.15 ms and 48.9 -> 47.7 ms); eight rows and one token
// at a time otherwise (with two, each token's q / k / g rows are loaded four
// times as often: 6.7 -> 11.6 ms for 64 units of 8192).
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

    static_assert(ROWS == 8, "eight value rows per warp");
    auto reduce = [&](float (&d)[ROWS]) { warp_sum8(d, lane); };
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
        *reinterpret_cast<uint4*>(o + tok * VD + v0) = *reinterpret_cast<const uint4*>(o2);
    }
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
                    rec_token<ROWS>(cur, o, scale, l2norm, (size_t)(bos + t) * H + h, v0, lane, s);
                    after(t);
                }
            }
        }
    }
}

// Four tokens at once on this warp's two value rows (the exact recompute).
// With S the state before the window, D_i the decay from there through token
// i (the product of exp(g) over tokens 0 .. i) and F_ij = D_i / D_j (the
// product over tokens j+1 .. i, so no division and no range limit), the
// per-token rule unrolls to
//   delta_i = beta_i (v_i - (k_i D_i).S - sum_{j<i} c_ij delta_j),
//   o_i     = (q_i D_i).S + sum_{j<=i} d_ij delta_j,
//   S'      = D_3 S + sum_j (k_j F_3j) delta_j^T,
// c_ij = sum k_i k_j F_ij, d_ij = sum q_i k_j F_ij.  All 32 dot products of
// the window go through one warp reduction (a reduce-scatter, then the totals
// through shared memory) instead of one reduction per token.  Tokens n .. 3
// of a last partial window are inert (beta = 0, no decay, no output).
__device__ __forceinline__ void rec_window4(const TokIn<2> (&in)[4], int n, uint16_t* __restrict__ o, float scale,
                                            bool l2norm, size_t tok0, int H, int v0, int lane, float (&s)[2][4],
                                            float* red) {
    float qv[4][4], kv[4][4], e[4][4], bt[4], vv[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool ok = i < n;
        qv[i][0] = __uint_as_float(in[i].q.x << 16); qv[i][1] = __uint_as_float(in[i].q.x & 0xffff0000u);
        qv[i][2] = __uint_as_float(in[i].q.y << 16); qv[i][3] = __uint_as_float(in[i].q.y & 0xffff0000u);
        kv[i][0] = __uint_as_float(in[i].k.x << 16); kv[i][1] = __uint_as_float(in[i].k.x & 0xffff0000u);
        kv[i][2] = __uint_as_float(in[i].k.y << 16); kv[i][3] = __uint_as_float(in[i].k.y & 0xffff0000u);
        e[i][0] = ok ? __expf(in[i].g.x) : 1.f;
        e[i][1] = ok ? __expf(in[i].g.y) : 1.f;
        e[i][2] = ok ? __expf(in[i].g.z) : 1.f;
        e[i][3] = ok ? __expf(in[i].g.w) : 1.f;
        bt[i] = ok ? in[i].beta : 0.f;
        vv[i][0] = ok ? __uint_as_float(in[i].v[0] << 16) : 0.f;
        vv[i][1] = ok ? __uint_as_float(in[i].v[0] & 0xffff0000u) : 0.f;
        if (!ok) {
#pragma unroll
            for (int x = 0; x < 4; ++x) qv[i][x] = kv[i][x] = 0.f;
        }
    }
    float ks[4] = {1.f, 1.f, 1.f, 1.f}, qs[4] = {scale, scale, scale, scale};
    if (l2norm) {   // x / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
        float nr[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            nr[i] = kv[i][0] * kv[i][0] + kv[i][1] * kv[i][1] + kv[i][2] * kv[i][2] + kv[i][3] * kv[i][3];
            nr[4 + i] = qv[i][0] * qv[i][0] + qv[i][1] * qv[i][1] + qv[i][2] * qv[i][2] + qv[i][3] * qv[i][3];
        }
        warp_sum8(nr, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ks[i] = rsqrtf(nr[i] + 1e-6f);
            qs[i] = scale * rsqrtf(nr[4 + i] + 1e-6f);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            kv[i][x] *= ks[i];
            qv[i][x] *= qs[i];
        }
    // decays: D_i (from the window start), F_ij (j < i)
    float D[4][4], F10[4], F20[4], F21[4], F30[4], F31[4], F32[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        D[0][x] = e[0][x];
        D[1][x] = D[0][x] * e[1][x];
        D[2][x] = D[1][x] * e[2][x];
        D[3][x] = D[2][x] * e[3][x];
        F10[x] = e[1][x];
        F21[x] = e[2][x];
        F32[x] = e[3][x];
        F20[x] = e[1][x] * e[2][x];
        F31[x] = e[2][x] * e[3][x];
        F30[x] = F20[x] * e[3][x];
    }
    // this lane's parts of the 32 dot products:
    //   [2i + r] (k_i D_i).s_r, [8 + 2i + r] (q_i D_i).s_r,
    //   [16 ..] c_10 c_20 c_21 c_30 c_31 c_32, [22 ..] d_00 d_10 d_11 d_20 d_21 d_22 d_30 d_31 d_32 d_33
    float a[32];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float ak = 0.f, aq = 0.f;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                ak = fmaf(kv[i][x] * D[i][x], s[r][x], ak);
                aq = fmaf(qv[i][x] * D[i][x], s[r][x], aq);
            }
            a[2 * i + r] = ak;
            a[8 + 2 * i + r] = aq;
        }
    auto dot3 = [&](const float (&u)[4], const float (&w)[4], const float (&f)[4]) {
        return u[0] * w[0] * f[0] + u[1] * w[1] * f[1] + u[2] * w[2] * f[2] + u[3] * w[3] * f[3];
    };
    auto dot2 = [&](const float (&u)[4], const float (&w)[4]) {
        return u[0] * w[0] + u[1] * w[1] + u[2] * w[2] + u[3] * w[3];
    };
    a[16] = dot3(kv[1], kv[0], F10);
    a[17] = dot3(kv[2], kv[0], F20);
    a[18] = dot3(kv[2], kv[1], F21);
    a[19] = dot3(kv[3], kv[0], F30);
    a[20] = dot3(kv[3], kv[1], F31);
    a[21] = dot3(kv[3], kv[2], F32);
    a[22] = dot2(qv[0], kv[0]);
    a[23] = dot3(qv[1], kv[0], F10);
    a[24] = dot2(qv[1], kv[1]);
    a[25] = dot3(qv[2], kv[0], F20);
    a[26] = dot3(qv[2], kv[1], F21);
    a[27] = dot2(qv[2], kv[2]);
    a[28] = dot3(qv[3], kv[0], F30);
    a[29] = dot3(qv[3], kv[1], F31);
    a[30] = dot3(qv[3], kv[2], F32);
    a[31] = dot2(qv[3], kv[3]);
    // reduce-scatter by halving: after the five exchanges lane l holds the
    // warp total of entry l
    {
        float b16[16], b8[8], b4[4], b2[2];
        const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2, h1 = lane & 1;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            b16[j] = (h16 ? a[j + 16] : a[j]) + __shfl_xor_sync(0xffffffffu, h16 ? a[j] : a[j + 16], 16);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            b8[j] = (h8 ? b16[j + 8] : b16[j]) + __shfl_xor_sync(0xffffffffu, h8 ? b16[j] : b16[j + 8], 8);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b4[j] = (h4 ? b8[j + 4] : b8[j]) + __shfl_xor_sync(0xffffffffu, h4 ? b8[j] : b8[j + 4], 4);
#pragma unroll
        for (int j = 0; j < 2; ++j)
            b2[j] = (h2 ? b4[j + 2] : b4[j]) + __shfl_xor_sync(0xffffffffu, h2 ? b4[j] : b4[j + 2], 2);
        const float t = (h1 ? b2[1] : b2[0]) + __shfl_xor_sync(0xffffffffu, h1 ? b2[0] : b2[1], 1);
        red[lane] = t;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 t = *reinterpret_cast<const float4*>(red + j);
        a[j] = t.x; a[j + 1] = t.y; a[j + 2] = t.z; a[j + 3] = t.w;
    }
    __syncwarp();   // every lane has read the totals before the next window writes them
    // the four deltas and outputs per value row
    float dl[4][2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        dl[0][r] = bt[0] * (vv[0][r] - a[r]);
        dl[1][r] = bt[1] * (vv[1][r] - a[2 + r] - a[16] * dl[0][r]);
        dl[2][r] = bt[2] * (vv[2][r] - a[4 + r] - a[17] * dl[0][r] - a[18] * dl[1][r]);
        dl[3][r] = bt[3] * (vv[3][r] - a[6 + r] - a[19] * dl[0][r] - a[20] * dl[1][r] - a[21] * dl[2][r]);
    }
    if (lane == 0) {
        float ov[4][2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            ov[0][r] = a[8 + r] + a[22] * dl[0][r];
            ov[1][r] = a[10 + r] + a[23] * dl[0][r] + a[24] * dl[1][r];
            ov[2][r] = a[12 + r] + a[25] * dl[0][r] + a[26] * dl[1][r] + a[27] * dl[2][r];
            ov[3][r] = a[14 + r] + a[28] * dl[0][r] + a[29] * dl[1][r] + a[30] * dl[2][r] + a[31] * dl[3][r];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i < n)
                *reinterpret_cast<__nv_bfloat162*>(o + (tok0 + (size_t)i * H) * VD + v0) =
                    __floats2bfloat162_rn(ov[i][0], ov[i][1]);
    }
    // state after the window
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            float y = D[3][x] * s[r][x];
            y = fmaf(kv[0][x] * F30[x], dl[0][r], y);
            y = fmaf(kv[1][x] * F31[x], dl[1][r], y);
            y = fmaf(kv[2][x] * F32[x], dl[2][r], y);
            y = fmaf(kv[3][x], dl[3][r], y);
            s[r][x] = y;
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
// recurrence is the same per-token rule (with two rows per warp, unrolled
// over windows of four tokens with exact pairwise decays), so it is exact
// for any decay.
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
    if constexpr (ROWS == 2) {
        // windows of four tokens, the next window's inputs loaded while the
        // current one is computed
        __shared__ __align__(16) float red_all[REC_THREADS];
        float* red = red_all + warp * 32;
        TokIn<2> cur[4], nxt[4];
        auto load_window = [&](TokIn<2> (&w)[4], int t0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + i < len) w[i] = load_tok<2>(p.q, p.k, p.v, p.g, p.beta, (size_t)(bos + t0 + i) * H + h, v0, lane);
        };
        load_window(cur, 0);
        for (int t0 = 0; t0 < len; t0 += 4) {
            if (t0 + 4 < len) load_window(nxt, t0 + 4);
            rec_window4(cur, len - t0 < 4 ? len - t0 : 4, p.o, p.scale, l2norm != 0, (size_t)(bos + t0) * H + h, H, v0,
                        lane, s, red);
#pragma unroll
            for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
        }
    } else {
        rec_tokens<ROWS, EXACT_AHEAD>(p.q, p.k, p.v, p.g, p.beta, p.o, p.scale, l2norm != 0, bos, len, H, h, v0, lane, s,
                                      [](int) {});
    }
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
