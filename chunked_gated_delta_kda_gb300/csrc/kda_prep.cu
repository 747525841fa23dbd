// Chunk-parallel half of the chunked KDA forward ("prep"): for one
// (chunk, head) it computes, from q, k, v, g, beta,
//   - the gate prefix sum G = cumsum(g) inside the chunk       (step M1)
//   - A  = beta_c * sum_d k_c k_i exp(G_c - G_i), i < c        (step M2)
//     A2 = sum_d (scale q_c) k_i exp(G_c - G_i),  i <= c        (M4's A2)
//   - (I + A)^-1 by blocked forward substitution, fp32        (step M2)
//   - w = (I+A)^-1 diag(beta)(exp(G) k), u = (I+A)^-1 diag(beta) v  (step M3)
//   - the transition-form tiles the sequential scan consumes:
//       Nm = -kg^T w, Bc = kg^T u, Qe = qg - A2 w, Oi = A2 u, Dg = exp(G_last)
//     (an exact re-association of step M4, see kda_common.cuh).
// Page: "PyPTO-Gym chunk_kda operator: an NPU forward of chunked gated
// delta-rule linear attention", section "算法原理" (M1-M4), "尾部 chunk 的零填充"
// (tail rows are zero: g = 0 keeps G flat so G_last is the last valid row,
// beta = 0 makes the rows inert), and "数值稳定性" (fp32 inverse; the gated
// products are factored around a pivot row with the exponent capped at 80).
//
// GB300 mapping.  One CTA of 256 threads per (chunk, head); the five
// 128-wide contractions run on tcgen05 tensor cores with fp32 accumulators in
// TMEM (A/A2 with bf16 operands for range, everything downstream of the
// inverse with fp16 operands for precision); elementwise work, the prefix sum
// and the small levels of the inverse run on CUDA cores in fp32.
#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int PREP_THREADS = 256;
constexpr float LOG2E = 1.4426950408889634f;
// exp2 argument cap: 2^115 ~ e^80, the page's decay cap; keeps every factor
// finite so that a zero operand never meets an infinite one.
constexpr float EXP2_CAP = 115.0f;

// Shared-memory map (bytes from the 1024-aligned base).
constexpr uint32_t RX = 0;        // 64 KB: Lk | Lq  ->  qg | kg
constexpr uint32_t RY = 65536;    // 32 KB: R  -> inverse temps -> merge tiles -> Ainv -> Nm staging
constexpr uint32_t RZ = 98304;    // 64 KB: RHS [t][k|v] -> w|u -> Qe | Oi staging
constexpr uint32_t RW = 163840;   // 48 KB: A (fp32, lower part) -> A2 fp16 -> Bc staging
constexpr uint32_t RM = 212992;   // misc
constexpr uint32_t M_G64 = RM;             // f32[128]  G at the pivot row (log2 units)
constexpr uint32_t M_GL = RM + 512;        // f32[128]  G at the last row (log2 units)
constexpr uint32_t M_BETA = RM + 1024;     // f32[128]
constexpr uint32_t M_INVQ = RM + 1536;     // f32[128]  scale / ||q|| (or scale)
constexpr uint32_t M_INVK = RM + 2048;     // f32[128]  1 / ||k|| (or 1)
constexpr uint32_t M_TOT = RM + 2560;      // f32[4][128] quarter sums of the scan
constexpr uint32_t M_DG = RM + 4608;       // f32[128]  exp(G_last) staging (bulk store)
constexpr uint32_t M_BAR = RM + 5120;      // mbarriers
constexpr uint32_t M_TMEM = RM + 5184;     // TMEM base address
constexpr uint32_t M_FLAG = RM + 5188;     // failure flag
constexpr uint32_t SMEM_USED = RM + 5248;
constexpr uint32_t PREP_SMEM = SMEM_USED + 1024;  // + alignment slack

// fp32 lower-triangular store of A in region W: columns 0..63 for all rows,
// columns 64..127 only for rows 64..127.  16-byte chunks XOR-swizzled by row.
__device__ __forceinline__ uint32_t as_off(int r, int c) {
    const uint32_t base = (c < 64) ? (uint32_t)r * 256u : 32768u + (uint32_t)(r - 64) * 256u;
    const int cc = c & 63;
    return base + (uint32_t)(((cc >> 2) ^ (r & 15)) << 4) + (uint32_t)(cc & 3) * 4u;
}

__device__ __forceinline__ float lds_f(const uint8_t* s, uint32_t off) {
    return *reinterpret_cast<const float*>(s + off);
}
__device__ __forceinline__ void sts_f(uint8_t* s, uint32_t off, float x) {
    *reinterpret_cast<float*>(s + off) = x;
}
__device__ __forceinline__ void sts_u32(uint8_t* s, uint32_t off, uint32_t x) {
    *reinterpret_cast<uint32_t*>(s + off) = x;
}
__device__ __forceinline__ void sts_v4(uint8_t* s, uint32_t off, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    *reinterpret_cast<uint4*>(s + off) = make_uint4(a, b, c, d);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t ldg_u32(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ float2 ldg_f2(const float* p) { return __ldg(reinterpret_cast<const float2*>(p)); }

// Issue one 128-row MMA over K = 16 * ksteps.  Descriptor start addresses
// advance per k-step by `a_step` / `b_step` bytes inside a slab and by the
// slab stride every 4 k-steps for K-major operands.
struct Operand {
    uint32_t base;
    bool mn_major;
    uint32_t rows;    // rows of one slab (K-major: M or N extent; MN-major: K extent)
};

__device__ __forceinline__ uint64_t op_desc(const Operand& o, int ks) {
    if (o.mn_major) {
        // MN-major 128B swizzle: K rows of 128 B, 8-row groups 1024 B apart,
        // 64-wide MN atoms one slab (rows * 128 B) apart.
        return smem_desc(o.base + (uint32_t)ks * 2048u, o.rows * 128u, 1024u, SW_128B);
    }
    // K-major 128B swizzle: M/N rows of 128 B, K advances 32 B per k-step
    // inside a 64-wide slab.
    return smem_desc(o.base + (uint32_t)(ks >> 2) * o.rows * 128u + (uint32_t)(ks & 3) * 32u, 16u, 1024u,
                     SW_128B);
}

__device__ __forceinline__ void mma_128(uint32_t d_tmem, const Operand& a, const Operand& b, uint32_t idesc,
                                        int ksteps) {
    for (int ks = 0; ks < ksteps; ++ks) mma_f16(d_tmem, op_desc(a, ks), op_desc(b, ks), idesc, ks > 0);
}

}  // namespace

template <bool L2NORM>
__global__ void __launch_bounds__(PREP_THREADS, 1) kda_prep_kernel(const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);

    ChunkRef c;
    if (!slot_chunk(p, (int)blockIdx.x, c)) return;   // uniform: no chunk in this slot
    const int h = (int)blockIdx.y;
    const int H = p.H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int len = c.len;

    float* sG64 = reinterpret_cast<float*>(sm + M_G64);
    float* sGL = reinterpret_cast<float*>(sm + M_GL);
    float* sBeta = reinterpret_cast<float*>(sm + M_BETA);
    float* sInvQ = reinterpret_cast<float*>(sm + M_INVQ);
    float* sInvK = reinterpret_cast<float*>(sm + M_INVK);
    float* sTot = reinterpret_cast<float*>(sm + M_TOT);
    float* sDg = reinterpret_cast<float*>(sm + M_DG);
    const uint32_t bar = sbase + M_BAR;
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(sm + M_FLAG);
    uint32_t phase = 0;

    if (warp == 0) {
        tmem_alloc(sbase + M_TMEM, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sFlag = 0;
    }
    const size_t row0 = (size_t)c.tok0 * H + h;  // row index of token tok0, head h
    if (tid < BT) {
        sBeta[tid] = tid < len ? __ldg(p.beta + row0 + (size_t)tid * H) : 0.f;
        if (!L2NORM) {
            sInvQ[tid] = p.scale;
            sInvK[tid] = 1.f;
        }
    }
    if (L2NORM) {
        // per-row 1/sqrt(sum x^2 + 1e-6), one warp per row
        for (int t = warp; t < BT; t += PREP_THREADS / 32) {
            float sq = 0.f, sk = 0.f;
            if (t < len) {
                const size_t off = (row0 + (size_t)t * H) * KD + lane * 4;
                const uint2 qv = __ldg(reinterpret_cast<const uint2*>(p.q + off));
                const uint2 kv = __ldg(reinterpret_cast<const uint2*>(p.k + off));
                float2 a = unpack_bf16(qv.x), b = unpack_bf16(qv.y);
                sq = a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y;
                a = unpack_bf16(kv.x);
                b = unpack_bf16(kv.y);
                sk = a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y;
            }
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, s);
                sk += __shfl_xor_sync(0xffffffffu, sk, s);
            }
            if (lane == 0) {
                sInvQ[t] = p.scale * rsqrtf(sq + 1e-6f);
                sInvK[t] = rsqrtf(sk + 1e-6f);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + M_TMEM);

    // ------------------------------------------------------------------
    // Phase 1: prefix sum of the gate over the chunk (log2 units), pivot at
    // row 64, operands of the gated products.  Thread = (d-pair, quarter).
    // ------------------------------------------------------------------
    const int pr = tid & 63;
    const int d0 = pr * 2;
    const int qtr = tid >> 6;
    const int tq0 = qtr * 32;
    float G0[32], G1[32];
    {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int t = tq0 + r;
            float2 gv = make_float2(0.f, 0.f);
            if (t < len) gv = ldg_f2(p.g + (row0 + (size_t)t * H) * KD + d0);
            a0 += gv.x * LOG2E;
            a1 += gv.y * LOG2E;
            G0[r] = a0;
            G1[r] = a1;
        }
        sTot[qtr * 128 + d0] = a0;
        sTot[qtr * 128 + d0 + 1] = a1;
    }
    __syncthreads();
    {
        float o0 = 0.f, o1 = 0.f;
        for (int q2 = 0; q2 < qtr; ++q2) {
            o0 += sTot[q2 * 128 + d0];
            o1 += sTot[q2 * 128 + d0 + 1];
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            G0[r] += o0;
            G1[r] += o1;
        }
        if (qtr == 2) {
            sG64[d0] = G0[0];
            sG64[d0 + 1] = G1[0];
        }
        if (qtr == 3) {
            sGL[d0] = G0[31];
            sGL[d0 + 1] = G1[31];
        }
    }
    __syncthreads();
    const float P0 = sG64[d0], P1 = sG64[d0 + 1];
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const int t = tq0 + r;
        float2 kf = make_float2(0.f, 0.f), qf = make_float2(0.f, 0.f);
        if (t < len) {
            const size_t off = (row0 + (size_t)t * H) * KD + d0;
            kf = unpack_bf16(ldg_u32(p.k + off));
            qf = unpack_bf16(ldg_u32(p.q + off));
        }
        const float ik = sInvK[t], iq = sInvQ[t];
        kf.x *= ik; kf.y *= ik;
        qf.x *= iq; qf.y *= iq;
        const float E0 = exp2f(fminf(G0[r] - P0, EXP2_CAP)), E1 = exp2f(fminf(G1[r] - P1, EXP2_CAP));
        const float F0 = exp2f(fminf(P0 - G0[r], EXP2_CAP)), F1 = exp2f(fminf(P1 - G1[r], EXP2_CAP));
        const uint32_t off = sw128_off(t, d0, 128);
        sts_u32(sm, RX + off, pack_bf16(kf.x * E0, kf.y * E1));            // Lk
        sts_u32(sm, RX + 32768 + off, pack_bf16(qf.x * E0, qf.y * E1));    // Lq
        sts_u32(sm, RY + off, pack_bf16(kf.x * F0, kf.y * F1));            // R
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint32_t id = idesc_f16(T_BF16, 128, 128, false, false);
        const Operand Lk{sbase + RX, false, 128}, Lq{sbase + RX + 32768, false, 128}, R{sbase + RY, false, 128};
        mma_128(tmem + 0, Lk, R, id, 8);     // A_raw  -> cols [0,128)
        mma_128(tmem + 128, Lq, R, id, 8);   // A2_raw -> cols [128,256)
        mma_commit(bar);
    }

    // ------------------------------------------------------------------
    // Phase 2 (after the gated products are done with their operands):
    // RHS = [beta exp(G) k | beta v] (fp16, MN-major [t][n]) in Z,
    // qg = scale q exp(G) and kg = k exp(G_last - G) (fp16) in X.
    // ------------------------------------------------------------------
    if (!mbar_wait(bar, phase, WAIT_LIMIT)) *sFlag = 1;
    phase ^= 1;
    tc_fence_after();
    {
        const float eP0 = exp2f(P0), eP1 = exp2f(P1);
        const float cL0 = exp2f(fminf(sGL[d0] - P0, EXP2_CAP)), cL1 = exp2f(fminf(sGL[d0 + 1] - P1, EXP2_CAP));
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int t = tq0 + r;
            float2 kf = make_float2(0.f, 0.f), qf = make_float2(0.f, 0.f), vf = make_float2(0.f, 0.f);
            if (t < len) {
                const size_t off = (row0 + (size_t)t * H) * KD + d0;
                kf = unpack_bf16(ldg_u32(p.k + off));
                qf = unpack_bf16(ldg_u32(p.q + off));
                vf = unpack_bf16(ldg_u32(p.v + off));
            }
            const float ik = sInvK[t], iq = sInvQ[t], b = sBeta[t];
            kf.x *= ik; kf.y *= ik;
            qf.x *= iq; qf.y *= iq;
            const float E0 = exp2f(fminf(G0[r] - P0, EXP2_CAP)), E1 = exp2f(fminf(G1[r] - P1, EXP2_CAP));
            const float F0 = exp2f(fminf(P0 - G0[r], EXP2_CAP)), F1 = exp2f(fminf(P1 - G1[r], EXP2_CAP));
            const float eg0 = E0 * eP0, eg1 = E1 * eP1;     // exp(G_t), <= 1
            const uint32_t off = sw128_off(t, d0, 128);
            sts_u32(sm, RZ + off, pack_f16(b * kf.x * eg0, b * kf.y * eg1));                 // RHS k part
            sts_u32(sm, RZ + sw128_off(t, 128 + d0, 128), pack_f16(b * vf.x, b * vf.y));     // RHS v part
            sts_u32(sm, RX + off, pack_f16(qf.x * eg0, qf.y * eg1));                         // qg
            sts_u32(sm, RX + 32768 + off, pack_f16(kf.x * F0 * cL0, kf.y * F1 * cL1));       // kg
        }
        if (qtr == 0) {
            sDg[d0] = exp2f(sGL[d0]);
            sDg[d0 + 1] = exp2f(sGL[d0 + 1]);
        }
    }

    // ------------------------------------------------------------------
    // Phase 3: A (strictly lower, times beta_row) from TMEM into fp32 smem,
    // then the blocked inverse of (I + A).
    // ------------------------------------------------------------------
    {
        const int row = (warp & 3) * 32 + lane;
        const int hc = warp >> 2;      // column half this warp reads
        if (!(hc == 1 && row < 64)) {
            const float b = sBeta[row];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                const int col0 = hc * 64 + part * 32;
                tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col0, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const int cc = col0 + j;
                    float a0 = (cc + 0 < row) ? b * x[j + 0] : 0.f;
                    float a1 = (cc + 1 < row) ? b * x[j + 1] : 0.f;
                    float a2 = (cc + 2 < row) ? b * x[j + 2] : 0.f;
                    float a3 = (cc + 3 < row) ? b * x[j + 3] : 0.f;
                    *reinterpret_cast<float4*>(sm + RW + as_off(row, cc)) = make_float4(a0, a1, a2, a3);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // Level 0: inverses of the eight 16x16 diagonal blocks, one column per
    // thread, by forward substitution (unit diagonal implied).
    {
        float x[16];
        const int blk = tid >> 4, j = tid & 15;
        if (tid < 128) {
            const int r0 = blk * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < i; ++m) s += lds_f(sm + RW, as_off(r0 + i, r0 + m)) * x[m];
                x[i] = (i == j) ? 1.f : (i < j ? 0.f : -s);
            }
        }
        __syncthreads();
        if (tid < 128) {
            const int r0 = blk * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i > j) sts_f(sm + RW, as_off(r0 + i, r0 + j), x[i]);
        }
        __syncthreads();
    }
    // Levels 1 and 2: merge pairs of inverted diagonal blocks,
    //   inv([[X, 0], [Y, Z]]) = [[Xi, 0], [-Zi Y Xi, Zi]],
    // first T = Y Xi into a temp (region Y), then -Zi T in place of Y.
    // Stored blocks hold only strictly-lower entries; the unit diagonal is
    // added where used.
    {
        float* tmp = reinterpret_cast<float*>(sm + RY);
        // level 1: 4 merges of 16-blocks; level 2: 2 merges of 32-blocks.
#pragma unroll
        for (int lvl = 1; lvl <= 2; ++lvl) {
            const int bs = lvl == 1 ? 16 : 32;              // size of the blocks being merged
            const int nmerge = lvl == 1 ? 4 : 2;
            const int per = bs * bs / (PREP_THREADS / nmerge);   // outputs per thread: 4 or 8
            const int tpm = PREP_THREADS / nmerge;          // threads per merge
            const int m = tid / tpm;
            const int li = tid % tpm;
            const int rr = li / (bs / per);                 // output row inside the block
            const int cc0 = (li % (bs / per)) * per;        // first output column
            const int C0 = m * 2 * bs;                      // first row/col of Xi
            const int R0 = C0 + bs;                         // first row of Y / Zi
            float acc[8];
            // T = Y Xi
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            for (int mm = 0; mm < bs; ++mm) {
                const float y = lds_f(sm + RW, as_off(R0 + rr, C0 + mm));
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (e < per) {
                        const int col = cc0 + e;
                        const float xv = (mm == col) ? 1.f : (mm > col ? lds_f(sm + RW, as_off(C0 + mm, C0 + col)) : 0.f);
                        acc[e] += y * xv;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < per) tmp[m * bs * bs + rr * bs + cc0 + e] = acc[e];
            __syncthreads();
            // L = -Zi T
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            for (int mm = 0; mm <= rr; ++mm) {
                const float z = (mm == rr) ? 1.f : lds_f(sm + RW, as_off(R0 + rr, R0 + mm));
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < per) acc[e] += z * tmp[m * bs * bs + mm * bs + cc0 + e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < per) sts_f(sm + RW, as_off(R0 + rr, C0 + cc0 + e), -acc[e]);
            __syncthreads();
        }
    }
    // Level 3 on tensor cores: L = -Q (A10 P) with P = inv of rows/cols
    // 0..63, Q = inv of rows/cols 64..127.  fp16 tiles in region Y:
    //   A10h [r][m] K-major (rows 64..127 of the M=128 MMA read the next tile
    //   and land in TMEM lanes that are never read), P_h [m][c] MN-major,
    //   Q_h [r'][r] K-major, T_h [r][c] MN-major; each 64 x 64, 8 KB.
    {
        constexpr uint32_t YA = RY, YP = RY + 8192, YQ = RY + 16384, YT = RY + 24576;
        for (int idx = tid; idx < 64 * 32; idx += PREP_THREADS) {
            const int r = idx >> 5, c2 = (idx & 31) * 2;     // element pair (r, c2), (r, c2+1)
            const float a0 = lds_f(sm + RW, as_off(64 + r, c2)), a1 = lds_f(sm + RW, as_off(64 + r, c2 + 1));
            sts_u32(sm, YA + sw128_off(r, c2, 64), pack_f16(a0, a1));
            float p0 = lds_f(sm + RW, as_off(r, c2)) + (r == c2 ? 1.f : 0.f);
            float p1 = lds_f(sm + RW, as_off(r, c2 + 1)) + (r == c2 + 1 ? 1.f : 0.f);
            sts_u32(sm, YP + sw128_off(r, c2, 64), pack_f16(p0, p1));
            float q0 = lds_f(sm + RW, as_off(64 + r, 64 + c2)) + (r == c2 ? 1.f : 0.f);
            float q1 = lds_f(sm + RW, as_off(64 + r, 64 + c2 + 1)) + (r == c2 + 1 ? 1.f : 0.f);
            sts_u32(sm, YQ + sw128_off(r, c2, 64), pack_f16(q0, q1));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const Operand A10{sbase + YA, false, 64}, Ph{sbase + YP, true, 64};
            mma_128(tmem + 0, A10, Ph, idesc_f16(T_F16, 128, 64, false, true), 4);   // T -> cols [0,64)
            mma_commit(bar);
        }
        if (!mbar_wait(bar, phase, WAIT_LIMIT)) *sFlag = 1;
        phase ^= 1;
        tc_fence_after();
        if ((warp & 3) < 2) {
            const int r = (warp & 3) * 32 + lane;            // T row (0..63)
            const int col0 = (warp >> 2) * 32;
            float x[32];
            tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col0, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                sts_v4(sm, YT + sw128_off(r, col0 + j, 64), pack_f16(x[j], x[j + 1]), pack_f16(x[j + 2], x[j + 3]),
                       pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const Operand Qh{sbase + YQ, false, 64}, Th{sbase + YT, true, 64};
            mma_128(tmem + 64, Qh, Th, idesc_f16(T_F16, 128, 64, false, true, /*neg_a=*/true), 4);  // L -> cols [64,128)
            mma_commit(bar);
        }
        if (!mbar_wait(bar, phase, WAIT_LIMIT)) *sFlag = 1;
        phase ^= 1;
        tc_fence_after();
        // L (fp32) replaces A10 in the fp32 store.
        if ((warp & 3) < 2) {
            const int r = (warp & 3) * 32 + lane;
            const int col0 = (warp >> 2) * 32;
            float x[32];
            tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 64u + (uint32_t)col0, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(sm + RW + as_off(64 + r, col0 + j)) =
                    make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
        }
        tc_fence_before();
        __syncthreads();
    }
    // Assemble (I + A)^-1 as fp16, K-major [c][i], in region Y.
    for (int ch = tid; ch < 128 * 16; ch += PREP_THREADS) {
        const int r = ch >> 4, c0 = (ch & 15) * 8;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int cc = c0 + e;
            float val = 0.f;
            if (!(r < 64 && cc >= 64)) val = lds_f(sm + RW, as_off(r, cc));
            x[e] = val + (cc == r ? 1.f : 0.f);
        }
        sts_v4(sm, RY + sw128_off(r, c0, 128), pack_f16(x[0], x[1]), pack_f16(x[2], x[3]), pack_f16(x[4], x[5]),
               pack_f16(x[6], x[7]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ------------------------------------------------------------------
    // Phase 4: [w | u] = Ainv [beta exp(G) k | beta v]  (M=128, N=256, K=128)
    // ------------------------------------------------------------------
    if (tid == 0) {
        const Operand Ai{sbase + RY, false, 128}, Rh{sbase + RZ, true, 128};
        mma_128(tmem + 256, Ai, Rh, idesc_f16(T_F16, 128, 256, false, true), 8);
        mma_commit(bar);
    }
    // Meanwhile: A2 (inclusive lower) from TMEM cols [128,256) to fp16
    // K-major [t][i] in region W (the fp32 store is no longer needed).
    {
        const int row = (warp & 3) * 32 + lane;
        const int col0 = (warp >> 2) * 64;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float x[32];
            const int cb = col0 + part * 32;
            tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 128u + (uint32_t)cb, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = (cb + j + e <= row) ? x[j + e] : 0.f;
                sts_v4(sm, RW + sw128_off(row, cb + j, 128), pack_f16(y[0], y[1]), pack_f16(y[2], y[3]),
                       pack_f16(y[4], y[5]), pack_f16(y[6], y[7]));
            }
        }
    }
    if (!mbar_wait(bar, phase, WAIT_LIMIT)) *sFlag = 1;
    phase ^= 1;
    tc_fence_after();

    // ------------------------------------------------------------------
    // Phase 5: w | u from TMEM cols [256,512) to fp16 MN-major [t][n] in Z.
    // ------------------------------------------------------------------
    {
        const int row = (warp & 3) * 32 + lane;
        const int col0 = (warp >> 2) * 128;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float x[32];
            const int cb = col0 + part * 32;
            tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 256u + (uint32_t)cb, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                sts_v4(sm, RZ + sw128_off(row, cb + j, 128), pack_f16(x[j], x[j + 1]), pack_f16(x[j + 2], x[j + 3]),
                       pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ------------------------------------------------------------------
    // Phase 6: [kg^T w | kg^T u] -> cols [0,256);  [A2 w | A2 u] -> [256,512)
    // ------------------------------------------------------------------
    if (tid == 0) {
        const Operand KgT{sbase + RX + 32768, true, 128}, A2h{sbase + RW, false, 128}, WU{sbase + RZ, true, 128};
        mma_128(tmem + 0, KgT, WU, idesc_f16(T_F16, 128, 256, true, true), 8);
        mma_128(tmem + 256, A2h, WU, idesc_f16(T_F16, 128, 256, false, true), 8);
        mma_commit(bar);
    }
    if (!mbar_wait(bar, phase, WAIT_LIMIT)) *sFlag = 1;
    phase ^= 1;
    tc_fence_after();

    // ------------------------------------------------------------------
    // Phase 7: epilogue into staging, then bulk stores to the workspace.
    //   warps 0-3: lanes = d;  Nm = -(kg^T w) -> Y,  Bc = kg^T u -> W
    //   warps 4-7: lanes = t;  Qe = qg - A2 w -> Z[0,32K), Oi = A2 u -> Z[32K,64K)
    // ------------------------------------------------------------------
    {
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        if (warp < 4) {
#pragma unroll 1
            for (int part = 0; part < 8; ++part) {
                float x[32];
                tmem_ld32(tmem + lane_off + (uint32_t)(part * 32), x);
                tmem_ld_wait();
                if (part < 4) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        const int cc = part * 32 + j;
                        sts_v4(sm, RY + sw128_off(row, cc, 128), pack_f16(-x[j], -x[j + 1]),
                               pack_f16(-x[j + 2], -x[j + 3]), pack_f16(-x[j + 4], -x[j + 5]),
                               pack_f16(-x[j + 6], -x[j + 7]));
                    }
                } else {
                    const int vt = part - 4;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, RW + vt * BC_PIECE + sw64_off(row, j), pack_f16(x[j], x[j + 1]),
                               pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
                }
            }
        } else {
#pragma unroll 1
            for (int part = 0; part < 8; ++part) {
                float x[32];
                tmem_ld32(tmem + lane_off + 256u + (uint32_t)(part * 32), x);
                tmem_ld_wait();
                if (part < 4) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        const int cc = part * 32 + j;
                        const uint4 qv = *reinterpret_cast<const uint4*>(sm + RX + sw128_off(row, cc, 128));
                        const float2 g0 = unpack_f16(qv.x), g1 = unpack_f16(qv.y), g2 = unpack_f16(qv.z),
                                     g3 = unpack_f16(qv.w);
                        // Qe goes to Z[0,32K), which held w|u: all MMAs reading it are done.
                        sts_v4(sm, RZ + sw128_off(row, cc, 128), pack_f16(g0.x - x[j], g0.y - x[j + 1]),
                               pack_f16(g1.x - x[j + 2], g1.y - x[j + 3]), pack_f16(g2.x - x[j + 4], g2.y - x[j + 5]),
                               pack_f16(g3.x - x[j + 6], g3.y - x[j + 7]));
                    }
                } else {
                    const int vt = part - 4;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, RZ + 32768 + vt * OI_PIECE + sw64_off(row, j), pack_f16(x[j], x[j + 1]),
                               pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
                }
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *sFlag == 0) {
        uint8_t* dst = tile_ptr(p, c.slot, h);
        bulk_s2g(dst + TILE_NM, sbase + RY, KD * KD * 2);
        bulk_s2g(dst + TILE_QE, sbase + RZ, BT * KD * 2);
        bulk_s2g(dst + TILE_BC, sbase + RW, NVT * BC_PIECE);
        bulk_s2g(dst + TILE_OI, sbase + RZ + 32768, NVT * OI_PIECE);
        bulk_s2g(dst + TILE_DG, sbase + M_DG, KD * 4);
        bulk_commit();
        bulk_wait0();
    }
    if (tid == 0 && *sFlag != 0) atomicOr(p.status, STATUS_TIMEOUT);
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Host-side launcher.
cudaError_t launch_prep(const FwdParams& p, bool l2norm, cudaStream_t stream) {
    const dim3 grid((unsigned)p.nslots, (unsigned)p.H);
    cudaError_t e;
    if (l2norm) {
        e = cudaFuncSetAttribute(kda_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
        if (e != cudaSuccess) return e;
        kda_prep_kernel<true><<<grid, PREP_THREADS, PREP_SMEM, stream>>>(p);
    } else {
        e = cudaFuncSetAttribute(kda_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
        if (e != cudaSuccess) return e;
        kda_prep_kernel<false><<<grid, PREP_THREADS, PREP_SMEM, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace kda
