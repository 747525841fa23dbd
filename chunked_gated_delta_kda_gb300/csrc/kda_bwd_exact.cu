// Token-by-token KDA backward: gradients of <do, o> + <dht, ht> with respect
// to q, k, v, g, beta and h0, evaluated exactly (fp32) for any gate decay.
//
// Forward rule (page "PyPTO-Gym chunk_kda operator: an NPU forward of chunked
// gated delta-rule linear attention", section "算子定位与算法背景"), in the
// [V, K] state layout where every value row v is independent:
//   a_v = exp(g) * s_v;  r_v = v_v - k.a_v;  s_v' = a_v + beta r_v k;
//   o_v = q.s_v'                      (q carries the scale)
// The pages name the backward kernels but give no formulas; the chain rule
// through one token, with G_v = dL/ds_v' + do_v q, is
//   dq   = sum_v do_v s_v'            dv_v = beta (G_v.k)
//   dk   = beta sum_v (r_v G_v - (G_v.k) a_v)
//   dbeta = sum_v r_v (G_v.k)
//   dA_v = G_v - beta (G_v.k) k;  dg = sum_v dA_v * a_v;  dL/ds_v = exp(g) * dA_v
//
// One CTA owns one (sequence, head) at a time (a persistent loop over them):
// 16 warps x 8 value rows, each lane 4 consecutive K entries of each row, so
// every thread reads and writes only its own 32 state entries.  Pass 1 runs
// the forward over the sequence and stores the state entering every
// 128-token chunk; pass 2 walks the chunks backwards, recomputes the states
// entering each token of the chunk into a per-CTA scratch, then steps the
// token rule above backwards.  The sums over value rows (dq, dk, dg, dbeta)
// are reduced across warps through shared memory, one barrier per token.
// Each warp stages the inputs of its next token (and in the backward walk
// the state entering it) in shared memory by asynchronous copies while it
// computes the current one, so the dependent chain does not wait on global
// memory.  With q/k normalisation the kernel produces the gradients with respect to
// the normalised q and k; kda_l2norm_bwd_kernel applies the normalisation's
// chain rule afterwards.
#include <cuda_bf16.h>

#include "kda.h"
#include "kda_common.cuh"
#include "kda_bwd.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int XB_THREADS = 512;
constexpr int XB_WARPS = XB_THREADS / 32;
constexpr int XB_ROWS = 8;                        // value rows per warp
constexpr int XB_RED = 3 * KD + 4;                // dq, dk, dg partials + dbeta (padded)
constexpr uint32_t XB_RED_BYTES = 2u * XB_WARPS * XB_RED * 4u;
// One token's staging slot per warp (bytes): q, k (8 B per lane), g (16 B
// per lane), the warp's 8 value entries of v and of dout, beta, then the
// state entering the token (8 rows x 32 lanes x 16 B; backward walk only).
constexpr uint32_t SL_Q = 0, SL_K = 256, SL_G = 512, SL_V = 1024, SL_DO = 1040, SL_BETA = 1056, SL_S = 1152;
constexpr uint32_t SLOT_BYTES = SL_S + XB_ROWS * 32 * 16;   // 5248
constexpr uint32_t XB_SMEM = XB_RED_BYTES + 2u * XB_WARPS * SLOT_BYTES;
static_assert(XB_SMEM <= 232448, "shared memory above the 227 KB limit");

struct TokenIn {
    float q[4], k[4], e[4];   // this lane's K entries: scaled (normalised) q, (normalised) k, exp(g)
    float beta;
    float v[XB_ROWS];         // the warp's 8 value rows
};

__device__ __forceinline__ void load_rows8_bf16(const uint16_t* p, float (&x)[XB_ROWS]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage token tok's inputs (and, with state != null, the warp's rows of the
// state entering it) into a slot: one commit group per call.
__device__ __forceinline__ void stage_token(const BwdParams& p, size_t tok, int v0, int lane, uint32_t slot,
                                            bool with_dout, const float* state) {
    cp_async8(slot + SL_Q + 8u * lane, p.q + tok * KD + 4 * lane);
    cp_async8(slot + SL_K + 8u * lane, p.k + tok * KD + 4 * lane);
    cp_async16(slot + SL_G + 16u * lane, p.g + tok * KD + 4 * lane);
    if (lane == 0) {
        cp_async16(slot + SL_V, p.v + tok * VD + v0);
        if (with_dout) cp_async16(slot + SL_DO, p.dout + tok * VD + v0);
        cp_async4(slot + SL_BETA, p.beta + tok);
    }
    if (state != nullptr) {
#pragma unroll
        for (int r = 0; r < XB_ROWS; ++r) cp_async16(slot + SL_S + (uint32_t)(r * 32 + lane) * 16u, state + (size_t)r * KD + 4 * lane);
    }
    cp_commit();
}

// A staged token's inputs: unpacked, scaled (and normalised), exp(g)
__device__ __forceinline__ void read_token(const BwdParams& p, const uint8_t* slot, int lane, TokenIn& in) {
    load4_bf16(reinterpret_cast<const uint16_t*>(slot + SL_Q + 8 * lane), in.q);
    load4_bf16(reinterpret_cast<const uint16_t*>(slot + SL_K + 8 * lane), in.k);
    const float4 gv = *reinterpret_cast<const float4*>(slot + SL_G + 16 * lane);
    in.beta = *reinterpret_cast<const float*>(slot + SL_BETA);
    load_rows8_bf16(reinterpret_cast<const uint16_t*>(slot + SL_V), in.v);
    float qs = p.scale, ks = 1.f;
    if (p.l2norm) {   // x / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
        const float sq = warp_sum(in.q[0] * in.q[0] + in.q[1] * in.q[1] + in.q[2] * in.q[2] + in.q[3] * in.q[3]);
        const float sk = warp_sum(in.k[0] * in.k[0] + in.k[1] * in.k[1] + in.k[2] * in.k[2] + in.k[3] * in.k[3]);
        qs *= rsqrtf(sq + 1e-6f);
        ks = rsqrtf(sk + 1e-6f);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        in.q[i] *= qs;
        in.k[i] *= ks;
    }
    in.e[0] = __expf(gv.x); in.e[1] = __expf(gv.y); in.e[2] = __expf(gv.z); in.e[3] = __expf(gv.w);
}

// Forward token rule on the warp's rows (no read-out).
__device__ __forceinline__ void forward_token(const TokenIn& in, int lane, float (&s)[XB_ROWS][4]) {
    float dot[XB_ROWS];
#pragma unroll
    for (int r = 0; r < XB_ROWS; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[r][i] *= in.e[i];
            acc = fmaf(in.k[i], s[r][i], acc);
        }
        dot[r] = acc;
    }
    warp_sum8(dot, lane);
#pragma unroll
    for (int r = 0; r < XB_ROWS; ++r) {
        const float delta = in.beta * (in.v[r] - dot[r]);
#pragma unroll
        for (int i = 0; i < 4; ++i) s[r][i] = fmaf(in.k[i], delta, s[r][i]);
    }
}

__device__ __forceinline__ void load_state(const float* src, int lane, float (&s)[XB_ROWS][4]) {
#pragma unroll
    for (int r = 0; r < XB_ROWS; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(src + (size_t)r * KD + 4 * lane);
        s[r][0] = x.x; s[r][1] = x.y; s[r][2] = x.z; s[r][3] = x.w;
    }
}

__device__ __forceinline__ void store_state(float* dst, int lane, const float (&s)[XB_ROWS][4]) {
#pragma unroll
    for (int r = 0; r < XB_ROWS; ++r)
        *reinterpret_cast<float4*>(dst + (size_t)r * KD + 4 * lane) = make_float4(s[r][0], s[r][1], s[r][2], s[r][3]);
}

}  // namespace

__global__ void __launch_bounds__(XB_THREADS, 1)
kda_bwd_exact_kernel(const BwdParams p, const uint32_t* only) {
    extern __shared__ __align__(16) float red[];   // [2][XB_WARPS][XB_RED], then the staging slots
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* slots = reinterpret_cast<uint8_t*>(red) + XB_RED_BYTES + (size_t)warp * 2 * SLOT_BYTES;
    const uint32_t slots_s = smem_u32(slots);
    const int v0 = warp * XB_ROWS;
    const int H = p.H;
    const int units = p.N * H;
    float* scratch = p.scratch + (size_t)blockIdx.x * BT * VD * KD;

    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        if (only != nullptr && only[u] == 0u) continue;   // uniform
        const int n = u / H, h = u % H;
        long long bos;
        int len;
        if (p.cu == nullptr) {
            bos = (long long)n * p.T;
            len = p.T;
        } else {
            const int a = p.cu[n], b = p.cu[n + 1];
            if (a < 0 || b < a || b > p.T || (n == 0 && a != 0) || (n == p.N - 1 && b != p.T)) {
                if (threadIdx.x == 0) atomicOr(p.status, STATUS_BAD_CU);
                continue;
            }
            bos = a;
            len = b - a;
        }
        const int nch = (len + BT - 1) / BT;
        const size_t st = (((size_t)n * H + h) * VD + v0) * KD;
        __syncthreads();   // the previous unit's last reduction has been read

        // pass 1: forward, storing the state entering each chunk
        float s[XB_ROWS][4];
        if (p.h0 != nullptr) {
            load_state(p.h0 + st, lane, s);
        } else {
#pragma unroll
            for (int r = 0; r < XB_ROWS; ++r) s[r][0] = s[r][1] = s[r][2] = s[r][3] = 0.f;
        }
        auto ckpt_of = [&](int j) {
            const int slot = p.cu == nullptr ? n * p.NT + j : p.cu[n] / BT + n + j;
            return p.ckpt + (((size_t)slot * H + h) * VD + v0) * KD;
        };
        {
            // the tokens of every chunk but the last (replayed in pass 2),
            // each staged one token ahead
            const int tend = nch > 0 ? (nch - 1) * BT : 0;
            if (tend > 0) stage_token(p, (size_t)bos * H + h, v0, lane, slots_s, false, nullptr);
            for (int t = 0; t < tend; ++t) {
                if (t % BT == 0) store_state(ckpt_of(t / BT), lane, s);
                if (t + 1 < tend) {
                    stage_token(p, (size_t)(bos + t + 1) * H + h, v0, lane, slots_s + (uint32_t)((t + 1) & 1) * SLOT_BYTES,
                                false, nullptr);
                    cp_wait<1>();
                } else {
                    cp_wait<0>();
                }
                __syncwarp();
                TokenIn in;
                read_token(p, slots + (size_t)(t & 1) * SLOT_BYTES, lane, in);
                forward_token(in, lane, s);
                __syncwarp();   // the slot is read before the next stage overwrites it
            }
            if (nch > 0) store_state(ckpt_of(nch - 1), lane, s);
        }

        // pass 2: backward, chunk by chunk from the last
        float d[XB_ROWS][4];   // dL / d(state after the current token)
        if (p.dht != nullptr) {
            load_state(p.dht + st, lane, d);
        } else {
#pragma unroll
            for (int r = 0; r < XB_ROWS; ++r) d[r][0] = d[r][1] = d[r][2] = d[r][3] = 0.f;
        }
        for (int j = nch - 1; j >= 0; --j) {
            const int slot = p.cu == nullptr ? n * p.NT + j : p.cu[n] / BT + n + j;
            const int t0 = j * BT;
            const int t1 = min(len, t0 + BT);
            load_state(p.ckpt + (((size_t)slot * H + h) * VD + v0) * KD, lane, s);
            stage_token(p, (size_t)(bos + t0) * H + h, v0, lane, slots_s, false, nullptr);
            for (int t = t0; t < t1; ++t) {   // states entering each token of the chunk
                store_state(scratch + ((size_t)(t - t0) * VD + v0) * KD, lane, s);
                if (t + 1 < t1) {
                    stage_token(p, (size_t)(bos + t + 1) * H + h, v0, lane,
                                slots_s + (uint32_t)((t + 1 - t0) & 1) * SLOT_BYTES, false, nullptr);
                    cp_wait<1>();
                } else {
                    cp_wait<0>();
                }
                __syncwarp();
                TokenIn in;
                read_token(p, slots + (size_t)((t - t0) & 1) * SLOT_BYTES, lane, in);
                forward_token(in, lane, s);
                __syncwarp();
            }
            // the scratch states stored above are read back below by copies
            // this thread issues: its stores are ordered before them
            __threadfence_block();
            auto stage_back = [&](int t, int k) {   // token t with its state and dout, into slot k
                stage_token(p, (size_t)(bos + t) * H + h, v0, lane, slots_s + (uint32_t)k * SLOT_BYTES, true,
                            scratch + ((size_t)(t - t0) * VD + v0) * KD);
            };
            stage_back(t1 - 1, 0);
            for (int t = t1 - 1; t >= t0; --t) {
                const size_t tok = (size_t)(bos + t) * H + h;
                const int k = (t1 - 1 - t) & 1;
                if (t - 1 >= t0) {
                    stage_back(t - 1, k ^ 1);
                    cp_wait<1>();
                } else {
                    cp_wait<0>();
                }
                __syncwarp();
                const uint8_t* sl = slots + (size_t)k * SLOT_BYTES;
                TokenIn in;
                read_token(p, sl, lane, in);
                float dov[XB_ROWS];
                load_rows8_bf16(reinterpret_cast<const uint16_t*>(sl + SL_DO), dov);
                float a[XB_ROWS][4];
#pragma unroll
                for (int r = 0; r < XB_ROWS; ++r) {
                    const float4 x = *reinterpret_cast<const float4*>(sl + SL_S + (r * 32 + lane) * 16);
                    a[r][0] = x.x; a[r][1] = x.y; a[r][2] = x.z; a[r][3] = x.w;
                }
                __syncwarp();   // the slot is read before the next stage overwrites it

                float rr[XB_ROWS], gk[XB_ROWS];
#pragma unroll
                for (int r = 0; r < XB_ROWS; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a[r][i] *= in.e[i];
                        acc = fmaf(in.k[i], a[r][i], acc);
                    }
                    rr[r] = acc;
                }
                warp_sum8(rr, lane);
                float pdq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int r = 0; r < XB_ROWS; ++r) {
                    rr[r] = in.v[r] - rr[r];
                    const float br = in.beta * rr[r];
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pdq[i] = fmaf(dov[r], fmaf(in.k[i], br, a[r][i]), pdq[i]);   // do_v s_v'
                        d[r][i] = fmaf(dov[r], in.q[i], d[r][i]);                     // G_v
                        acc = fmaf(d[r][i], in.k[i], acc);
                    }
                    gk[r] = acc;
                }
                warp_sum8(gk, lane);
                float pdk[4] = {0.f, 0.f, 0.f, 0.f}, pdg[4] = {0.f, 0.f, 0.f, 0.f};
                float pdb = 0.f;
#pragma unroll
                for (int r = 0; r < XB_ROWS; ++r) {
                    pdb = fmaf(rr[r], gk[r], pdb);
                    const float bg = in.beta * gk[r];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pdk[i] = fmaf(rr[r], d[r][i], fmaf(-gk[r], a[r][i], pdk[i]));
                        d[r][i] = fmaf(-bg, in.k[i], d[r][i]);                      // dA_v
                        pdg[i] = fmaf(d[r][i], a[r][i], pdg[i]);
                        d[r][i] *= in.e[i];                                           // dL/ds_v (previous)
                    }
                }
                if (lane < 2) {   // dv_v = beta (G_v.k), rows v0 + 4 lane .. + 3
                    const int r0 = 4 * lane;
                    *reinterpret_cast<float4*>(p.dv + tok * VD + v0 + r0) =
                        make_float4(in.beta * gk[r0], in.beta * gk[r0 + 1], in.beta * gk[r0 + 2], in.beta * gk[r0 + 3]);
                }
                float* buf = red + ((size_t)(t & 1) * XB_WARPS + warp) * XB_RED;
                *reinterpret_cast<float4*>(buf + 4 * lane) = make_float4(pdq[0], pdq[1], pdq[2], pdq[3]);
                *reinterpret_cast<float4*>(buf + KD + 4 * lane) = make_float4(pdk[0], pdk[1], pdk[2], pdk[3]);
                *reinterpret_cast<float4*>(buf + 2 * KD + 4 * lane) = make_float4(pdg[0], pdg[1], pdg[2], pdg[3]);
                if (lane == 0) buf[3 * KD] = pdb;
                __syncthreads();
                const int i = threadIdx.x;
                if (i <= 3 * KD) {
                    const float* col = red + (size_t)(t & 1) * XB_WARPS * XB_RED + i;
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < XB_WARPS; ++w) sum += col[(size_t)w * XB_RED];
                    if (i < KD) p.dq[tok * KD + i] = p.scale * sum;
                    else if (i < 2 * KD) p.dk[tok * KD + i - KD] = in.beta * sum;
                    else if (i < 3 * KD) p.dg[tok * KD + i - 2 * KD] = sum;
                    else p.dbeta[tok] = sum;
                }
            }
        }
        if (p.dh0 != nullptr) store_state(p.dh0 + st, lane, d);
    }
}

// Chain rule of the per-token normalisation x_hat = x / sqrt(|x|^2 + 1e-6):
// dx = (dx_hat - x_hat (x_hat . dx_hat)) / sqrt(|x|^2 + 1e-6), in place on
// dq and dk (one warp per (token, head)).
__global__ void __launch_bounds__(256) kda_l2norm_bwd_kernel(const uint16_t* __restrict__ q,
                                                             const uint16_t* __restrict__ k, float* dq, float* dk,
                                                             long long rows) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    for (int which = 0; which < 2; ++which) {
        const uint16_t* x = which == 0 ? q : k;
        float* dx = which == 0 ? dq : dk;
        float xv[4];
        load4_bf16(x + (size_t)row * KD + 4 * lane, xv);
        float4 d = *reinterpret_cast<const float4*>(dx + (size_t)row * KD + 4 * lane);
        const float inv = rsqrtf(warp_sum(xv[0] * xv[0] + xv[1] * xv[1] + xv[2] * xv[2] + xv[3] * xv[3]) + 1e-6f);
        const float dot = warp_sum((xv[0] * d.x + xv[1] * d.y + xv[2] * d.z + xv[3] * d.w) * inv);
        d.x = (d.x - xv[0] * inv * dot) * inv;
        d.y = (d.y - xv[1] * inv * dot) * inv;
        d.z = (d.z - xv[2] * inv * dot) * inv;
        d.w = (d.w - xv[3] * inv * dot) * inv;
        *reinterpret_cast<float4*>(dx + (size_t)row * KD + 4 * lane) = d;
    }
}

cudaError_t launch_bwd_exact(const BwdParams& p, const uint32_t* only, int ctas, cudaStream_t stream) {
    if (p.N == 0 || ctas == 0) return cudaSuccess;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(kda_bwd_exact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)XB_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    kda_bwd_exact_kernel<<<ctas, XB_THREADS, XB_SMEM, stream>>>(p, only);
    return cudaGetLastError();
}

cudaError_t launch_l2norm_bwd(const BwdParams& p, long long rows, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    kda_l2norm_bwd_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p.q, p.k, p.dq, p.dk, rows);
    return cudaGetLastError();
}

}  // namespace kda
