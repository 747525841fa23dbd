// Chunk-parallel KDA backward on the tensor cores: the chunked form of the
// per-token chain rule (the same gradients as kda_bwd_chunk_kernel).
//
// Per 128-token chunk with entering state S0 (K x V), exit state gradient Z
// and n valid rows, with G the in-chunk inclusive prefix sum of g and a pivot
// P = G at row min(n - 1, 64) (the pivot of the forward's chunk-parallel
// kernel, section "算法原理" of the page "PyPTO-Gym chunk_kda operator: an NPU
// forward of chunked gated delta-rule linear attention"):
//   qh = scale q e^{G-P},  kh = k e^{G-P},  kc = k e^{P-G}
//   Sp = e^{P} S0 (rows),  Ze = e^{G_last - P} Z (rows)
//   Pm = strict_tril(kh kc^T),  Aqk = tril(qh kc^T),  Lb = I + diag(beta) Pm
//   y0 = v - kh Sp,  rho = Lb^{-1} diag(beta) y0          (rho_t = beta_t r_t)
// so that o = qh Sp + Aqk rho and the exit state is e^{G_last} S0 + (e^{G_last-P} kc)^T rho.
// Differentiating those products (P cancels from the loss and is held fixed):
//   W = tril(do rho^T),  drho = Aqk^T do + kc Ze,  dy = Lb^{-T} drho
//   X = strict_tril(dy rho^T)
//   dv = beta dy,  dbeta = rowsum(dy * y0) - rowsum(X * Pm)
//   dqh = do Sp^T + W kc
//   dkh = -diag(beta) dy Sp^T - diag(beta) X kc
//   dkc = W^T qh + rho Ze^T - X^T diag(beta) kh
//   dG = qh dqh + kh dkh - kc dkc, plus at the last row
//        colsum(kc * (rho Ze^T)) + e^{G_last} rowsum(Z * S0)
//   dg = reverse prefix sum of dG;  dq = scale dqh e^{G-P};  dk = dkh e^{G-P} + dkc e^{P-G}
// Every product is a 128 x 128 x 128 (or triangular) one, evaluated with
// warp-level TF32 tensor-core instructions (mma.sync m16n8k8, fp32
// accumulation; TF32 keeps fp32's exponent range, so the pivot-factored
// operands need no cap while the forward's factoring range holds).  The
// inverse of the unit lower-triangular Lb is blocked: 16 x 16 diagonal blocks
// by forward substitution, then merges 16 -> 32 -> 64 -> 128 with
// inv([[A, 0], [C, D]]) = [[A^-1, 0], [-D^-1 C A^-1, D^-1]].
//
// A chunk whose factors would leave fp32's range (in-chunk decay beyond e^60
// from the pivot row, or a pivot or exit decay below e^-60) is not computed
// here: it is marked in tc_skip for the per-token chunk kernel, which is exact
// for any decay.
//
// One CTA of 16 warps per chunk (persistent over chunks), three 128 x 132
// fp32 shared-memory operand buffers; every product's 128 x 128 result is one
// 32 x 32 tile per warp, held in registers until a barrier, so an epilogue
// may overwrite the buffers the product read.  Matrices needed again later
// live in a per-CTA global scratch (about 1 MB per CTA, mostly L2-resident).
#include <cuda_bf16.h>

#include "kda.h"
#include "kda_bwd.cuh"
#include "kda_common.cuh"
#include "sm100_ptx.cuh"
#include "kda_mma_tf32.cuh"
#include "kda_bwd_inv.cuh"

namespace kda {

namespace {

constexpr int TC_THREADS = 512;
constexpr int TC_WARPS = TC_THREADS / 32;
constexpr int LD = MMA_LD;                              // padded row length of the shared buffers
constexpr int MAT = BT * LD;                            // floats per shared buffer
constexpr int NVEC = 17;                                // 128-float vectors in shared memory (+ the TMEM address)
constexpr uint32_t TC_SMEM = (3u * MAT + NVEC * 128u) * 4u;
constexpr float TC_RANGE = 60.f;                        // |exponent| bound of the factored operands

// per-CTA global scratch: 128 x 128 fp32 matrices (row length 128)
enum : int { SC_QH = 0, SC_KH, SC_KC, SC_AQK, SC_PM, SC_LI, SC_Y0, SC_RHO, SC_W, SC_X, SC_COUNT };
// TMEM columns (each a 128-column block): matrices a warp keeps in its own
// fragment order (32 values per thread, lane 32 (warp % 4) + lane, columns
// 32 (warp / 4) .. + 31 of the block) instead of round-tripping global memory
constexpr uint32_t TM_G = 0, TM_DQH = 128, TM_DKH = 256, TM_DKC = 384, TM_COLS = 512;
constexpr size_t SC_MAT = (size_t)BT * 128;

// shared vectors
enum : int { V_BETA = 0, V_PIV, V_GLAST, V_EXIT, V_UNUSED, V_NQ, V_NK, V_TMP, V_TSLOT,
             V_DBP = 9,     // 4 vectors: dbeta partials of the four column-band warps (summed in a fixed order)
             V_EXP = 13 };  // 4 vectors: exit-term column partials of the four row-band warps

__device__ __forceinline__ float (&flat(float (&acc)[2][4][4]))[32] {
    return *reinterpret_cast<float(*)[32]>(&acc[0][0][0]);
}

__device__ __forceinline__ void zero_acc(float (&acc)[2][4][4]) {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) acc[mi][nj][0] = acc[mi][nj][1] = acc[mi][nj][2] = acc[mi][nj][3] = 0.f;
}

// Visit the elements of a warp's 32 x 32 tile: f(i, j, value).
template <class F>
__device__ __forceinline__ void tile_for(const float (&acc)[2][4][4], int i0, int j0, int lane, F f) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
            const int i = i0 + 16 * mi + g, j = j0 + 8 * nj + 2 * t;
            f(i, j, acc[mi][nj][0]);
            f(i, j + 1, acc[mi][nj][1]);
            f(i + 8, j, acc[mi][nj][2]);
            f(i + 8, j + 1, acc[mi][nj][3]);
        }
}

// The warp tile's elements as 16 pairs of row-adjacent columns: pair q = (mi * 4 + nj) * 2 + hh
// holds (i, j) and (i, j + 1) with i = i0 + 16 mi + g + 8 hh, j = j0 + 8 nj + 2 t, i.e.
// acc[mi][nj][2 hh] and acc[mi][nj][2 hh + 1].
template <class F>
__device__ __forceinline__ void frag_pairs(int i0, int j0, int lane, F f) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int nj = 0; nj < 4; ++nj)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) f((mi * 4 + nj) * 2 + hh, mi, nj, hh, i0 + 16 * mi + g + 8 * hh, j0 + 8 * nj + 2 * t);
}

// Full 128 x 128 x 128 product: warp w owns the tile at rows 32 (w / 4), cols 32 (w % 4).
template <bool TA, bool TB>
__device__ __forceinline__ void mm128(const float* A, const float* B, int warp, int lane, float (&acc)[2][4][4]) {
    tile_mm<TA, TB>(A, B, 32 * (warp >> 2), 32 * (warp & 3), BT, lane, acc);
}

// global (row length 128) <-> shared (row length LD), with an optional element transform
__device__ __forceinline__ void stage(float* dst, const float* __restrict__ src, int tid) {
#pragma unroll
    for (int i = tid; i < BT * 32; i += TC_THREADS) {
        const int r = i >> 5, c4 = (i & 31) * 4;
        *reinterpret_cast<float4*>(dst + r * LD + c4) = *reinterpret_cast<const float4*>(src + r * 128 + c4);
    }
}
// Stores of the gradients with an L2 evict-first policy: streamed once, they
// should not push the per-CTA scratch out of L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_ef(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_ef2(float* p, float a, float b, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(a), "f"(b), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_ef4(float* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void spill(float* dst, const float* src, int tid) {
#pragma unroll
    for (int i = tid; i < BT * 32; i += TC_THREADS) {
        const int r = i >> 5, c4 = (i & 31) * 4;
        *reinterpret_cast<float4*>(dst + r * 128 + c4) = *reinterpret_cast<const float4*>(src + r * LD + c4);
    }
}

__device__ __forceinline__ void bf16x8(const uint4 u, float (&x)[8]) {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}

// dst (shared) = the chunk's bf16 rows of src (token-major, rows row0 + r rs), zero past n
__device__ __forceinline__ void stage_rows_bf16(float* dst, const uint16_t* __restrict__ src, size_t row0, size_t rs,
                                                int n, int tid) {
#pragma unroll
    for (int i = tid; i < BT * 16; i += TC_THREADS) {
        const int r = i >> 4, c8 = (i & 15) * 8;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) u = *reinterpret_cast<const uint4*>(src + (row0 + r * rs) * 128 + c8);
        float x[8];
        bf16x8(u, x);
        *reinterpret_cast<float4*>(dst + r * LD + c8) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(dst + r * LD + c8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
}

// Last reads of the streamed inputs, with the same policy.
__device__ __forceinline__ uint4 ld_ef_u4(const void* p, uint64_t pol) {
    uint4 r;
    asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ float4 ld_ef_f4(const void* p, uint64_t pol) {
    float4 r;
    asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint32_t ld_ef_u32(const void* p, uint64_t pol) {
    uint32_t r;
    asm("ld.global.nc.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ void stage_rows_bf16_ef(float* dst, const uint16_t* __restrict__ src, size_t row0, size_t rs,
                                                   int n, int tid, uint64_t pol) {
#pragma unroll
    for (int i = tid; i < BT * 16; i += TC_THREADS) {
        const int r = i >> 4, c8 = (i & 15) * 8;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) u = ld_ef_u4(src + (row0 + r * rs) * 128 + c8, pol);
        float x[8];
        bf16x8(u, x);
        *reinterpret_cast<float4*>(dst + r * LD + c8) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(dst + r * LD + c8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
}

// stage_state_scaled with the evict-first policy (the state's last read)
__device__ __forceinline__ void stage_state_scaled_ef(float* dst, const float* __restrict__ src, const float* e, int tid,
                                                      uint64_t pol) {
#pragma unroll
    for (int i = tid; i < KD * 32; i += TC_THREADS) {
        const int r = i >> 5, c4 = (i & 31) * 4;
        float4 x = ld_ef_f4(src + r * VD + c4, pol);
        const float f = __expf(e[r]);
        x.x *= f; x.y *= f; x.z *= f; x.w *= f;
        *reinterpret_cast<float4*>(dst + r * LD + c4) = x;
    }
}

// dst (shared) = diag(exp(e[r])) src (a [K][V] fp32 state)
__device__ __forceinline__ void stage_state_scaled(float* dst, const float* __restrict__ src, const float* e, int tid) {
#pragma unroll
    for (int i = tid; i < KD * 32; i += TC_THREADS) {
        const int r = i >> 5, c4 = (i & 31) * 4;
        float4 x = *reinterpret_cast<const float4*>(src + r * VD + c4);
        const float f = __expf(e[r]);
        x.x *= f; x.y *= f; x.z *= f; x.w *= f;
        *reinterpret_cast<float4*>(dst + r * LD + c4) = x;
    }
}

}  // namespace

__global__ void __launch_bounds__(TC_THREADS, 1) kda_bwd_tc_kernel(const BwdParams p, const FwdParams fp) {
    extern __shared__ __align__(16) float tsm[];
    float* B0 = tsm;
    float* B1 = tsm + MAT;
    float* B2 = tsm + 2 * MAT;
    float* vec = tsm + 3 * MAT;
    float* vBeta = vec + V_BETA * 128;
    float* vPiv = vec + V_PIV * 128;
    float* vGl = vec + V_GLAST * 128;
    float* vExit = vec + V_EXIT * 128;
    float* vNq = vec + V_NQ * 128;
    float* vNk = vec + V_NK * 128;
    float* vTmp = vec + V_TMP * 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    const long long items = (long long)fp.nslots * H;
    float* sc = p.scratch + (size_t)blockIdx.x * BT * VD * KD;
    auto S = [&](int m) { return sc + (size_t)m * SC_MAT; };
    const int ti0 = 32 * (warp >> 2), tj0 = 32 * (warp & 3);   // this warp's output tile
    const float scale = p.scale;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(vec + V_TSLOT * 128);
    float* vDbP = vec + V_DBP * 128;   // [4][128]: [column band][row]
    float* vExP = vec + V_EXP * 128;   // [4][128]: [row band][column]
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
    // this thread's private 32 columns of each TMEM block
    const uint32_t tme = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32u * (uint32_t)(warp >> 2);
    auto tm_put = [&](uint32_t blk, float (&acc)[2][4][4]) {
        tmem_st32(tme + blk, flat(acc));
        tmem_st_wait();
    };
    auto tm_get = [&](uint32_t blk, float (&acc)[2][4][4]) {
        tmem_ld32(tme + blk, flat(acc));
        tmem_ld_wait();
    };

    const uint64_t efp = evict_first_policy();
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const int slot = (int)(it / H), h = (int)(it % H);
        ChunkRef c;
        if (!slot_chunk(fp, slot, c)) continue;                    // uniform
        if (fp.exact_flags[(size_t)c.n * H + h] != 0u) continue;   // replayed by the token-by-token kernel
        long long bos;
        int len;
        if (!seq_bounds(fp, c.n, bos, len)) continue;
        const int nch = (len + BT - 1) / BT;
        const int n = c.len;
        const int piv = n - 1 < 64 ? n - 1 : 64;
        const size_t row0 = (size_t)c.tok0 * H + h;                // (token, head) row of the chunk's first token
        const size_t rs = (size_t)H;                               // rows between tokens
        const float* S0 = p.ckpt_s + ((size_t)slot * H + h) * KD * VD;
        const float* Z = p.ckpt_d + ((size_t)chunk_slot(fp, c.n, nch - 1 - c.j) * H + h) * KD * VD;
        __syncthreads();   // the previous chunk's last reads of the shared buffers are done

        // ---- gate prefix sums G (B0), beta, q/k row norms -------------------------------
#pragma unroll
        for (int i = tid; i < BT * 32; i += TC_THREADS) {
            const int r = i >> 5, c4 = (i & 31) * 4;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < n) x = ld_ef_f4(p.g + (row0 + r * rs) * KD + c4, efp);
            *reinterpret_cast<float4*>(B0 + r * LD + c4) = x;
        }
        if (tid < BT) vBeta[tid] = tid < n ? p.beta[row0 + tid * rs] : 0.f;
        if (p.l2norm) {   // per-row inverse norms 1 / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
            for (int r = warp; r < BT; r += TC_WARPS) {
                float sq = 0.f, sk = 0.f;
                if (r < n) {
                    float xq[4], xk[4];
                    load4_bf16(p.q + (row0 + r * rs) * KD + 4 * lane, xq);
                    load4_bf16(p.k + (row0 + r * rs) * KD + 4 * lane, xk);
                    sq = xq[0] * xq[0] + xq[1] * xq[1] + xq[2] * xq[2] + xq[3] * xq[3];
                    sk = xk[0] * xk[0] + xk[1] * xk[1] + xk[2] * xk[2] + xk[3] * xk[3];
                }
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                if (lane == 0) {
                    vNq[r] = rsqrtf(sq + 1e-6f);
                    vNk[r] = rsqrtf(sk + 1e-6f);
                }
            }
        } else if (tid < BT) {
            vNq[tid] = 1.f;
            vNk[tid] = 1.f;
        }
        __syncthreads();
        if (tid < KD) {   // column prefix sums; rows past n hold G_last
            float acc = 0.f;
            for (int r = 0; r < BT; ++r) {
                if (r < n) acc += B0[r * LD + tid];
                B0[r * LD + tid] = acc;
            }
            vPiv[tid] = B0[piv * LD + tid];
            vGl[tid] = acc;
            vTmp[tid] = acc - vPiv[tid];
            vExit[tid] = 0.f;
        }
        __syncthreads();
        // Range guard: the factors e^{+-(G-P)}, e^{P} and e^{G_last-P} must stay well
        // inside fp32; a chunk beyond that is left to the per-token kernel.
        bool wide = false;
        for (int i = tid; i < n * KD; i += TC_THREADS) {
            const int r = i >> 7, d = i & 127;
            const float x = B0[r * LD + d] - vPiv[d];
            wide = wide || !(fabsf(x) <= TC_RANGE);
        }
        if (tid < KD) wide = wide || !(vPiv[tid] >= -TC_RANGE) || !(vGl[tid] - vPiv[tid] >= -TC_RANGE);
        if (__syncthreads_or(wide)) {
            if (tid == 0) p.tc_skip[it] = 1u;
            continue;
        }
        {   // G at this warp's fragment positions -> TMEM
            float gf[2][4][4];
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    const int i = ti0 + 16 * mi + g, j = tj0 + 8 * nj + 2 * t;
                    gf[mi][nj][0] = B0[i * LD + j];
                    gf[mi][nj][1] = B0[i * LD + j + 1];
                    gf[mi][nj][2] = B0[(i + 8) * LD + j];
                    gf[mi][nj][3] = B0[(i + 8) * LD + j + 1];
                }
            tm_put(TM_G, gf);
        }

        // ---- gated operands: B0 = qh, B1 = kh, B2 = kc -----------------------------------
#pragma unroll 2
        for (int i = tid; i < BT * 16; i += TC_THREADS) {
            const int r = i >> 4, c8 = (i & 15) * 8;
            uint4 uq = make_uint4(0u, 0u, 0u, 0u), uk = uq;
            if (r < n) {
                uq = *reinterpret_cast<const uint4*>(p.q + (row0 + r * rs) * KD + c8);
                uk = *reinterpret_cast<const uint4*>(p.k + (row0 + r * rs) * KD + c8);
            }
            float xq[8], xk[8];
            bf16x8(uq, xq);
            bf16x8(uk, xk);
            const float sq = vNq[r] * scale, sk = vNk[r];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int d = c8 + u;
                const float e = B0[r * LD + d] - vPiv[d];
                const float ep = __expf(e), em = __expf(-e);
                B1[r * LD + d] = xk[u] * sk * ep;
                B2[r * LD + d] = xk[u] * sk * em;
                B0[r * LD + d] = xq[u] * sq * ep;
            }
        }
        __syncthreads();
        spill(S(SC_QH), B0, tid);
        spill(S(SC_KH), B1, tid);
        spill(S(SC_KC), B2, tid);

        float acc[2][4][4];
        // ---- Aqk = tril(qh kc^T) -----------------------------------------------------------
        zero_acc(acc);
        mm128<false, true>(B0, B2, warp, lane, acc);
        tile_for(acc, ti0, tj0, lane, [&](int i, int j, float x) { S(SC_AQK)[i * 128 + j] = (j <= i) ? x : 0.f; });
        // ---- Pm = strict_tril(kh kc^T); B0 = Lb = I + diag(beta) Pm ------------------------
        zero_acc(acc);
        mm128<false, true>(B1, B2, warp, lane, acc);
        __syncthreads();
        tile_for(acc, ti0, tj0, lane, [&](int i, int j, float x) {
            const float pm = (j < i) ? x : 0.f;
            S(SC_PM)[i * 128 + j] = pm;
            B0[i * LD + j] = (i == j) ? 1.f : vBeta[i] * pm;
        });
        __syncthreads();
        invert_unit_lower(B0, warp, lane, tid);   // B0 = Li
        spill(S(SC_LI), B0, tid);
        // ---- B2 = Sp = e^P S0 (rows) ---------------------------------------------------------
        stage_state_scaled(B2, S0, vPiv, tid);
        __syncthreads();
        // ---- y0 = v - kh Sp; B1 = y = beta y0 (v fetched before the product) ---------------
        {
            uint32_t vpre[16];
            frag_pairs(ti0, tj0, lane, [&](int q, int, int, int, int i, int j) {
                vpre[q] = i < n ? ld_ef_u32(p.v + (row0 + i * rs) * VD + j, efp) : 0u;
            });
            zero_acc(acc);
            mm128<false, false>(B1, B2, warp, lane, acc);
            __syncthreads();
            frag_pairs(ti0, tj0, lane, [&](int q, int mi, int nj, int hh, int i, int j) {
                const float y0a = __uint_as_float(vpre[q] << 16) - acc[mi][nj][2 * hh];
                const float y0b = __uint_as_float(vpre[q] & 0xffff0000u) - acc[mi][nj][2 * hh + 1];
                *reinterpret_cast<float2*>(S(SC_Y0) + i * 128 + j) = make_float2(y0a, y0b);
                B1[i * LD + j] = vBeta[i] * y0a;
                B1[i * LD + j + 1] = vBeta[i] * y0b;
            });
        }
        __syncthreads();
        // ---- rho = Li y; B1 = rho ------------------------------------------------------------
        zero_acc(acc);
        mm128<false, false>(B0, B1, warp, lane, acc);
        __syncthreads();
        tile_for(acc, ti0, tj0, lane, [&](int i, int j, float x) {
            S(SC_RHO)[i * 128 + j] = x;
            B1[i * LD + j] = x;
        });
        // ---- B0 = do; W = tril(do rho^T) ---------------------------------------------------
        stage_rows_bf16(B0, p.dout, row0, rs, n, tid);
        __syncthreads();
        zero_acc(acc);
        mm128<false, true>(B0, B1, warp, lane, acc);
        tile_for(acc, ti0, tj0, lane, [&](int i, int j, float x) { S(SC_W)[i * 128 + j] = (j <= i) ? x : 0.f; });
        __syncthreads();
        // ---- drho = Aqk^T do + kc Ze --------------------------------------------------------
        stage(B1, S(SC_AQK), tid);
        __syncthreads();
        zero_acc(acc);
        mm128<true, false>(B1, B0, warp, lane, acc);
        __syncthreads();
        stage(B1, S(SC_KC), tid);
        {   // B2 = Ze = e^{G_last - P} Z (rows); the exit term e^{G_last} rowsum(Z * S0) on the way
            // step s of warp w covers state row w + 16 s (its 32 lanes x 4 columns)
            float part[8];
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const int r = warp + 16 * st, c4 = lane * 4;
                float4 zv = ld_ef_f4(Z + r * VD + c4, efp);
                const float4 sv = *reinterpret_cast<const float4*>(S0 + r * VD + c4);
                part[st] = zv.x * sv.x + zv.y * sv.y + zv.z * sv.z + zv.w * sv.w;
                const float f = __expf(vTmp[r]);
                zv.x *= f; zv.y *= f; zv.z *= f; zv.w *= f;
                *reinterpret_cast<float4*>(B2 + r * LD + c4) = zv;
            }
            warp_sum8(part, lane);
            if (lane == 0) {
#pragma unroll
                for (int st = 0; st < 8; ++st) vExit[warp + 16 * st] += __expf(vGl[warp + 16 * st]) * part[st];
            }
        }
        __syncthreads();
        mm128<false, false>(B1, B2, warp, lane, acc);
        __syncthreads();
        tile_for(acc, ti0, tj0, lane, [&](int i, int j, float x) { B1[i * LD + j] = x; });   // B1 = drho
        stage(B0, S(SC_LI), tid);
        __syncthreads();
        // ---- dy = Li^T drho; dv = beta dy; dbeta += rowsum(dy y0) --------------------------
        {
            float2 ypre[16];
            frag_pairs(ti0, tj0, lane, [&](int q, int, int, int, int i, int j) {
                ypre[q] = *reinterpret_cast<const float2*>(S(SC_Y0) + i * 128 + j);
            });
            zero_acc(acc);
            mm128<true, false>(B0, B1, warp, lane, acc);
            __syncthreads();
            float rsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            frag_pairs(ti0, tj0, lane, [&](int q, int mi, int nj, int hh, int i, int j) {
                const float a = acc[mi][nj][2 * hh], b = acc[mi][nj][2 * hh + 1];
                B1[i * LD + j] = a;
                B1[i * LD + j + 1] = b;
                if (i < n)
                    st_ef2(p.dv + (row0 + i * rs) * VD + j, vBeta[i] * a, vBeta[i] * b, efp);
                rsum[mi][hh] = fmaf(a, ypre[q].x, fmaf(b, ypre[q].y, rsum[mi][hh]));
            });
            // reduce over the 4 lanes sharing a row, then across the row band's warps
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    float v = rsum[mi][hi];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    if ((lane & 3) == 0) vDbP[(warp & 3) * 128 + ti0 + 16 * mi + 8 * hi + (lane >> 2)] = v;
                }
        }
        stage(B0, S(SC_RHO), tid);
        __syncthreads();
        // ---- X = strict_tril(dy rho^T); dbeta -= rowsum(X Pm) ------------------------------
        {
            float2 ppre[16];
            frag_pairs(ti0, tj0, lane, [&](int q, int, int, int, int i, int j) {
                ppre[q] = *reinterpret_cast<const float2*>(S(SC_PM) + i * 128 + j);
            });
            zero_acc(acc);
            mm128<false, true>(B1, B0, warp, lane, acc);
            float rsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            frag_pairs(ti0, tj0, lane, [&](int q, int mi, int nj, int hh, int i, int j) {
                const float a = (j < i) ? acc[mi][nj][2 * hh] : 0.f, b = (j + 1 < i) ? acc[mi][nj][2 * hh + 1] : 0.f;
                *reinterpret_cast<float2*>(S(SC_X) + i * 128 + j) = make_float2(a, b);
                rsum[mi][hh] = fmaf(-a, ppre[q].x, fmaf(-b, ppre[q].y, rsum[mi][hh]));
            });
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    float v = rsum[mi][hi];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    if ((lane & 3) == 0) vDbP[(warp & 3) * 128 + ti0 + 16 * mi + 8 * hi + (lane >> 2)] += v;
                }
        }
        // ---- dkc = rho Ze^T (+ later terms); exit term colsum(kc * rho Ze^T) ---------------
        {
            float2 kpre[16];
            frag_pairs(ti0, tj0, lane, [&](int q, int, int, int, int i, int j) {
                kpre[q] = *reinterpret_cast<const float2*>(S(SC_KC) + i * 128 + j);
            });
            zero_acc(acc);
            mm128<false, true>(B0, B2, warp, lane, acc);
            tm_put(TM_DKC, acc);
            float csum[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
            frag_pairs(ti0, tj0, lane, [&](int q, int mi, int nj, int hh, int, int) {
                csum[nj][0] = fmaf(kpre[q].x, acc[mi][nj][2 * hh], csum[nj][0]);
                csum[nj][1] = fmaf(kpre[q].y, acc[mi][nj][2 * hh + 1], csum[nj][1]);
            });
            // reduce over the 8 lanes sharing a column (lane / 4), then across warps
#pragma unroll
            for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                for (int lo = 0; lo < 2; ++lo) {
                    float v = csum[nj][lo];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    if (lane < 4) vExP[(warp >> 2) * 128 + tj0 + 8 * nj + 2 * lane + lo] = v;
                }
        }
        __syncthreads();
        // ---- B0 = Sp; dkh = -diag(beta) dy Sp^T -------------------------------------------
        stage_state_scaled_ef(B0, S0, vPiv, tid, efp);
        __syncthreads();
        zero_acc(acc);
        mm128<false, true>(B1, B0, warp, lane, acc);
        {
            const int g = lane >> 2;
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    const float b0 = -vBeta[ti0 + 16 * mi + g], b1 = -vBeta[ti0 + 16 * mi + g + 8];
                    acc[mi][nj][0] *= b0; acc[mi][nj][1] *= b0; acc[mi][nj][2] *= b1; acc[mi][nj][3] *= b1;
                }
            tm_put(TM_DKH, acc);
        }
        __syncthreads();
        // ---- B1 = do; dqh = do Sp^T ----------------------------------------------------------
        stage_rows_bf16_ef(B1, p.dout, row0, rs, n, tid, efp);
        __syncthreads();
        zero_acc(acc);
        mm128<false, true>(B1, B0, warp, lane, acc);
        __syncthreads();
        // ---- B0 = W, B2 = kc: dqh += W kc ------------------------------------------------
        stage(B0, S(SC_W), tid);
        stage(B2, S(SC_KC), tid);
        __syncthreads();
        mm128<false, false>(B0, B2, warp, lane, acc);
        tm_put(TM_DQH, acc);
        // ---- B1 = X: dkh -= diag(beta) X kc ---------------------------------------------
        __syncthreads();
        stage(B1, S(SC_X), tid);
        __syncthreads();
        zero_acc(acc);
        mm128<false, false>(B1, B2, warp, lane, acc);
        {
            float prev[2][4][4];
            tm_get(TM_DKH, prev);
            const int g = lane >> 2;
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int nj = 0; nj < 4; ++nj) {
                    const float b0 = vBeta[ti0 + 16 * mi + g], b1 = vBeta[ti0 + 16 * mi + g + 8];
                    prev[mi][nj][0] -= b0 * acc[mi][nj][0]; prev[mi][nj][1] -= b0 * acc[mi][nj][1];
                    prev[mi][nj][2] -= b1 * acc[mi][nj][2]; prev[mi][nj][3] -= b1 * acc[mi][nj][3];
                }
            tm_put(TM_DKH, prev);
        }
        // ---- B2 = qh: dkc += W^T qh ------------------------------------------------------
        __syncthreads();
        stage(B2, S(SC_QH), tid);
        __syncthreads();
        zero_acc(acc);
        mm128<true, false>(B0, B2, warp, lane, acc);
        __syncthreads();
        // ---- B0 = diag(beta) kh: dkc -= X^T (beta kh) ------------------------------------
#pragma unroll
        for (int i = tid; i < BT * 32; i += TC_THREADS) {
            const int r = i >> 5, c4 = (i & 31) * 4;
            float4 x = *reinterpret_cast<const float4*>(S(SC_KH) + r * 128 + c4);
            const float b = vBeta[r];
            x.x *= b; x.y *= b; x.z *= b; x.w *= b;
            *reinterpret_cast<float4*>(B0 + r * LD + c4) = x;
        }
        __syncthreads();
        {
            float acc2[2][4][4];
            zero_acc(acc2);
            mm128<true, false>(B1, B0, warp, lane, acc2);
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int nj = 0; nj < 4; ++nj)
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc[mi][nj][u] -= acc2[mi][nj][u];
        }
        {
            float prev[2][4][4];
            tm_get(TM_DKC, prev);
#pragma unroll
            for (int u = 0; u < 32; ++u) flat(prev)[u] += flat(acc)[u];
            tm_put(TM_DKC, prev);
        }
        __syncthreads();

        // ---- dG into B0; exit terms at the last row; reverse prefix sum; outputs -------------
        // raw q, k rows (B1, B2), then per fragment element from TMEM: dq, dk and dG (into B0)
        stage_rows_bf16_ef(B1, p.q, row0, rs, n, tid, efp);
        stage_rows_bf16_ef(B2, p.k, row0, rs, n, tid, efp);
        __syncthreads();
        {   // one 16-row half of the warp's tile at a time (fragment elements 16 mi .. 16 mi + 15)
            const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
            for (int mi = 0; mi < 2; ++mi) {
                float fg[16], fq[16], fh[16], fc[16];
                tmem_ld16(tme + TM_G + 16u * mi, fg);
                tmem_ld16(tme + TM_DQH + 16u * mi, fq);
                tmem_ld16(tme + TM_DKH + 16u * mi, fh);
                tmem_ld16(tme + TM_DKC + 16u * mi, fc);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int nj = e >> 2, u = e & 3;
                    const int i = ti0 + 16 * mi + g + 8 * (u >> 1), j = tj0 + 8 * nj + 2 * t + (u & 1);
                    const float x = fg[e] - vPiv[j];
                    const float ep = __expf(x), em = __expf(-x);
                    const float qq = scale * vNq[i] * B1[i * LD + j], kk = vNk[i] * B2[i * LD + j];
                    // dG = qh dqh + kh dkh - kc dkc
                    B0[i * LD + j] = qq * ep * fq[e] + kk * ep * fh[e] - kk * em * fc[e];
                    if (i < n) {   // with the q/k norm: w.r.t. the normalised q, k
                        st_ef(p.dq + (row0 + i * rs) * KD + j, scale * fq[e] * ep, efp);
                        st_ef(p.dk + (row0 + i * rs) * KD + j, fh[e] * ep + fc[e] * em, efp);
                    }
                }
            }
        }
        __syncthreads();
        if (tid < KD) {   // dg = reverse prefix sum over the valid rows, the exit terms at row n - 1
            float acc1 = vExit[tid] + ((vExP[tid] + vExP[128 + tid]) + (vExP[256 + tid] + vExP[384 + tid]));
            for (int r = n - 1; r >= 0; --r) {
                acc1 += B0[r * LD + tid];
                B0[r * LD + tid] = acc1;
            }
        }
        if (tid >= KD && tid < KD + BT && tid - KD < n) {
            const int r = tid - KD;
            p.dbeta[row0 + r * rs] = (vDbP[r] + vDbP[128 + r]) + (vDbP[256 + r] + vDbP[384 + r]);
        }
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < n * 32; i += TC_THREADS) {
            const int r = i >> 5, c4 = (i & 31) * 4;
            st_ef4(p.dg + (row0 + r * rs) * KD + c4, *reinterpret_cast<const float4*>(B0 + r * LD + c4), efp);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

cudaError_t launch_bwd_tc(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream) {
    if (fp.nslots == 0 || ctas == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    if (e != cudaSuccess) return e;
    kda_bwd_tc_kernel<<<ctas, TC_THREADS, TC_SMEM, stream>>>(p, fp);
    return cudaGetLastError();
}

}  // namespace kda
