// Chunk-parallel KDA backward on the 5th-generation tensor cores: the chunked
// form of the per-token chain rule (the same gradients and the same algebra as
// kda_bwd_tc_kernel, whose header sets it out) with every 128 x 128 x 128
// product a tcgen05.mma of kind::tf32 issued by one thread, operands read from
// shared memory through matrix descriptors and accumulators in TMEM.
//
// Operand layout.  Every operand is K-major: a matrix used as A (M x K) or as
// B (N x K) is stored row-major with the reduction index along the row, in
// the 128-byte-swizzled layout (four 32-column slabs of 128 rows x 128 bytes;
// within a 128-byte row the 16-byte chunk index is XORed with row % 8).  A
// product that needs a transposed operand gets it written transposed by the
// epilogue that produced it, or staged transposed from global memory, so the
// descriptors never use the transposed-operand mode.  Operands are rounded to
// TF32 (round to nearest) when stored.
//
// Accumulators: four 128-column TMEM blocks.  ACC takes the intermediate
// products (Aqk, y0, rho, W, drho, dy, X); DQH, DKH and DKC accumulate
//   dqh = do Sp^T + W kc,   -dkh / beta = dy Sp^T + X kc,
//   dkc = rho Ze^T + W^T qh - X^T (beta kh)
// across products (DKC also holds Pm briefly before its first product).
// Epilogues read one row per thread (warp w: TMEM lanes 32 (w % 4) .. + 31,
// columns 32 (w / 4) .. + 31), so row masks, row scalings and row sums are
// per-thread work.  Matrices needed again later live in a per-CTA global
// scratch; the unit lower-triangular inverse is the blocked one shared with
// the mma.sync kernel (on a padded fp32 copy).
//
// Selected by KDA_FLAG_BWD_UMMA.  On GB300 it is slower than the mma.sync
// kernel (20.9 against 16.5 ms for the per-chunk stage at T=65536, H=32):
// the products take ~15% of a chunk's cycles, the operand staging between
// them (gating, transposes, scratch round trips) the rest, with one chunk in
// flight per SM and nothing overlapping it.
#include <cuda_bf16.h>

#include "kda.h"
#include "kda_bwd.cuh"
#include "kda_bwd_inv.cuh"
#include "kda_common.cuh"
#include "kda_mma_tf32.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int UM_THREADS = 512;
constexpr int UM_WARPS = UM_THREADS / 32;
constexpr uint32_t SLOT = 69632;                      // one operand slot: 64 KiB swizzled, or 128 x 132 fp32 padded
constexpr int NV = 22;                                 // 128-float vectors after the slots
constexpr uint32_t UM_SMEM = 3u * SLOT + NV * 512u + 64u + 1024u;   // + barrier / TMEM word + alignment
constexpr float UM_RANGE = 60.f;

// per-CTA global scratch: plain row-major 128 x 128 fp32 matrices
enum : int { G_G = 0, G_QH, G_KH, G_KC, G_AQKT, G_PM, G_LI, G_Y0, G_RHO, G_W, G_WT, G_X, G_XT, G_COUNT };
constexpr size_t G_MAT = 128 * 128;
// TMEM blocks
constexpr uint32_t T_ACC = 0, T_DQH = 128, T_DKH = 256, T_DKC = 384, T_COLS = 512;
// shared vectors (128 floats each)
enum : int { V_BETA = 0, V_PIV, V_GLAST, V_TMP, V_NQ, V_NK,
             V_DBP = 6,     // 4: dbeta partials per column slice
             V_EXR = 10,    // 4: exit rowsum(Z * S0) partials per column block
             V_EXC = 14,    // 4: exit colsum(kc * rho Ze^T) partials per row quarter
             V_MISC = 18 };

__host__ __device__ constexpr uint32_t idesc_tf32_128() {
    return (1u << 4)            // D = f32
           | (2u << 7)          // A = tf32
           | (2u << 10)         // B = tf32
           | ((128u >> 3) << 17)
           | ((128u >> 4) << 24);
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A B^T over K = 128 for K-major swizzled A (128 x 128) and B (128 x 128)
// at shared addresses a, b: sixteen K = 8 steps, 32 bytes apart inside a
// 128-byte row, 16 KiB between the 32-column slabs.
__device__ __forceinline__ void umma128(uint32_t d_tmem, uint32_t a, uint32_t b, bool accumulate) {
    const uint64_t da = smem_desc(a, 16u, 1024u, SW_128B), db = smem_desc(b, 16u, 1024u, SW_128B);
    constexpr uint32_t id = idesc_tf32_128();
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
        const uint64_t step = (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2);   // 16-byte units
        umma_tf32(d_tmem, da + step, db + step, id, (ks > 0 || accumulate) ? 1u : 0u);
    }
}

// byte offset of element (r, c) of a K-major swizzled 128 x 128 fp32 operand
__device__ __forceinline__ uint32_t km(int r, int c) {
    return (uint32_t)((c >> 5) * 16384 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + (c & 3) * 4);
}

__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(to_tf32(x)); }

__device__ __forceinline__ void st_km4(uint8_t* slot, int r, int c4, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(slot + km(r, c4)) = make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}

__device__ __forceinline__ void bf16x8(const uint4 u, float (&x)[8]) {
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}

// Row r (32 floats from column 32 cs) of a plain row-major global matrix.
__device__ __forceinline__ void ld_row32(const float* __restrict__ src, int r, int cs, float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(src + (size_t)r * 128 + 32 * cs + 4 * q);
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
    }
}
__device__ __forceinline__ void st_row32(float* dst, int r, int cs, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(dst + (size_t)r * 128 + 32 * cs + 4 * q) =
            make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}
// transposed: element (r, 32 cs + c) -> dst[32 cs + c][r] (a warp's lanes write consecutive r)
__device__ __forceinline__ void st_rowT32(float* dst, int r, int cs, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 32; ++c) dst[(size_t)(32 * cs + c) * 128 + r] = x[c];
}
// into a K-major slot, same orientation / transposed
__device__ __forceinline__ void km_row32(uint8_t* slot, int r, int cs, const float (&x)[32]) {
#pragma unroll
    for (int q = 0; q < 8; ++q) st_km4(slot, r, 32 * cs + 4 * q, x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}
__device__ __forceinline__ void km_rowT32(uint8_t* slot, int r, int cs, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 32; ++c) *reinterpret_cast<float*>(slot + km(32 * cs + c, r)) = tf32r(x[c]);
}

// Stage a plain row-major global matrix into a K-major slot (row r scaled by scale(r)).
template <class F>
__device__ __forceinline__ void stage_km(uint8_t* slot, const float* __restrict__ src, int tid, F scale) {
#pragma unroll 4
    for (int i = tid; i < 128 * 32; i += UM_THREADS) {
        const int r = i >> 5, c4 = (i & 31) * 4;
        const float4 v = *reinterpret_cast<const float4*>(src + (size_t)r * 128 + c4);
        const float f = scale(r);
        st_km4(slot, r, c4, f * v.x, f * v.y, f * v.z, f * v.w);
    }
}
// Stage it transposed: source (r, c) -> slot (c, r), source row r scaled by scale(r).
// Warp w takes the 32 x 32 block of source rows 32 (w / 4) and columns 32 (w % 4);
// lane l holds source row 32 (w / 4) + l and writes one slot row segment per column.
template <class F>
__device__ __forceinline__ void stage_kmT(uint8_t* slot, const float* __restrict__ src, int warp, int lane, F scale) {
    const int r = 32 * (warp >> 2) + lane, cb = warp & 3;
    float x[32];
    ld_row32(src, r, cb, x);
    const float f = scale(r);
#pragma unroll
    for (int c = 0; c < 32; ++c) x[c] *= f;
    km_rowT32(slot, r, cb, x);
}

// The chunk's bf16 rows (token-major, row0 + t rs) into a K-major slot, same orientation or transposed.
__device__ __forceinline__ void stage_km_bf16(uint8_t* slot, const uint16_t* __restrict__ src, size_t row0, size_t rs,
                                              int n, int tid) {
#pragma unroll 2
    for (int i = tid; i < 128 * 16; i += UM_THREADS) {
        const int r = i >> 4, c8 = (i & 15) * 8;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) u = *reinterpret_cast<const uint4*>(src + (row0 + r * rs) * 128 + c8);
        float x[8];
        bf16x8(u, x);
        st_km4(slot, r, c8, x[0], x[1], x[2], x[3]);
        st_km4(slot, r, c8 + 4, x[4], x[5], x[6], x[7]);
    }
}
__device__ __forceinline__ void stage_kmT_bf16(uint8_t* slot, const uint16_t* __restrict__ src, size_t row0, size_t rs,
                                               int n, int warp, int lane) {
    const int r = 32 * (warp >> 2) + lane, cb = warp & 3;
    float x[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) u = *reinterpret_cast<const uint4*>(src + (row0 + r * rs) * 128 + 32 * cb + 8 * q);
        float y[8];
        bf16x8(u, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[8 * q + e] = y[e];
    }
    km_rowT32(slot, r, cb, x);
}

// Warp transpose-reduce: lane c ends with the sum over the 32 lanes of v[c] (31 shuffles).
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 32, m = 16; m >= 1; w >>= 1, m >>= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < w / 2; ++i) {
            const float send = up ? v[i] : v[i + w / 2];
            const float keep = up ? v[i + w / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    return v[0];
}

}  // namespace

__global__ void __launch_bounds__(UM_THREADS, 1) kda_bwd_umma_kernel(const BwdParams p, const FwdParams fp) {
    extern __shared__ uint8_t um_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(um_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* S0 = sm;
    uint8_t* S1 = sm + SLOT;
    uint8_t* S2 = sm + 2 * SLOT;
    float* vec = reinterpret_cast<float*>(sm + 3 * SLOT);
    float* vBeta = vec + V_BETA * 128;
    float* vPiv = vec + V_PIV * 128;
    float* vGl = vec + V_GLAST * 128;
    float* vTmp = vec + V_TMP * 128;
    float* vNq = vec + V_NQ * 128;
    float* vNk = vec + V_NK * 128;
    float* vDbP = vec + V_DBP * 128;
    float* vExR = vec + V_EXR * 128;
    float* vExC = vec + V_EXC * 128;
    uint8_t* misc = sm + 3 * SLOT + NV * 512u;
    const uint32_t bar = smem_u32(misc);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + 16);
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(misc + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qr = warp & 3, cs = warp >> 2;          // epilogue: row 32 qr + lane, columns 32 cs ..
    const int erow = 32 * qr + lane;
    const int H = p.H;
    const long long items = (long long)fp.nslots * H;
    float* sc = p.scratch + (size_t)blockIdx.x * BT * VD * KD;
    auto SG = [&](int m) { return sc + (size_t)m * G_MAT; };
    const float scale = p.scale;

    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), T_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sFlag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);
    const uint32_t trow = tmem + ((uint32_t)(32 * qr) << 16) + 32u * (uint32_t)cs;   // this thread's row segment
    uint32_t phase = 0;

    // operands written by the threads (and TMEM reads done) -> the tensor core may go
    auto to_mma = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    // bounded: once a wait of this CTA has run out, later ones return at once
    // and the item loop ends at its next iteration (tested right after a CTA
    // barrier, so every thread takes the same decision)
    const uint32_t wlim = wait_limit_of(fp);
    auto commit_wait = [&]() {
        if (tid == 0) mma_commit(bar);
        if (*sFlag == 0 && !mbar_wait(bar, phase, wlim)) *sFlag = 1;
        phase ^= 1u;
        tc_fence_after();
    };
    auto tm_row = [&](uint32_t blk, float (&x)[32]) {
        tmem_ld32(trow + blk, x);
        tmem_ld_wait();
    };

    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const int slot = (int)(it / H), h = (int)(it % H);
        ChunkRef c;
        if (!slot_chunk(fp, slot, c)) continue;
        if (fp.exact_flags[(size_t)c.n * H + h] != 0u) continue;
        long long bos;
        int len;
        if (!seq_bounds(fp, c.n, bos, len)) continue;
        const int nch = (len + BT - 1) / BT;
        const int n = c.len;
        const int piv = n - 1 < 64 ? n - 1 : 64;
        const size_t row0 = (size_t)c.tok0 * H + h;
        const size_t rs = (size_t)H;
        const float* Sc = p.ckpt_s + ((size_t)slot * H + h) * KD * VD;
        const float* Z = p.ckpt_d + ((size_t)chunk_slot(fp, c.n, nch - 1 - c.j) * H + h) * KD * VD;
        float* G0 = reinterpret_cast<float*>(S0);   // padded fp32 view (row length MMA_LD)
        tc_fence_before();
        __syncthreads();
        if (*sFlag != 0) break;

        // ---- gate prefix sums G (S0 padded), beta, q/k row norms --------------------------
#pragma unroll 4
        for (int i = tid; i < 128 * 32; i += UM_THREADS) {
            const int r = i >> 5, c4 = (i & 31) * 4;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < n) x = *reinterpret_cast<const float4*>(p.g + (row0 + r * rs) * KD + c4);
            *reinterpret_cast<float4*>(G0 + r * MMA_LD + c4) = x;
        }
        if (tid < BT) vBeta[tid] = tid < n ? p.beta[row0 + tid * rs] : 0.f;
        if (p.l2norm) {   // 1 / sqrt(sum x^2 + 1e-6) per row, section "测试与验证体系"
            for (int r = warp; r < BT; r += UM_WARPS) {
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
        if (tid < KD) {
            float acc = 0.f;
            for (int r = 0; r < BT; ++r) {
                if (r < n) acc += G0[r * MMA_LD + tid];
                G0[r * MMA_LD + tid] = acc;
            }
            vPiv[tid] = G0[piv * MMA_LD + tid];
            vGl[tid] = acc;
            vTmp[tid] = acc - vPiv[tid];
        }
        __syncthreads();
        bool wide = false;
        for (int i = tid; i < n * KD; i += UM_THREADS) {
            const int r = i >> 7, d = i & 127;
            wide = wide || !(fabsf(G0[r * MMA_LD + d] - vPiv[d]) <= UM_RANGE);
        }
        if (tid < KD) wide = wide || !(vPiv[tid] >= -UM_RANGE) || !(vTmp[tid] >= -UM_RANGE);
        if (__syncthreads_or(wide)) {
            if (tid == 0) p.tc_skip[it] = 1u;
            continue;
        }

        // ---- gated operands: kh -> S1, kc -> S2 (K-major); qh, kh, kc, G -> scratch ----------
        // (two 16-column halves of the thread's row segment)
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int c0 = 32 * cs + 16 * hf;
            float gq[16], q[16], k[16];
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) gq[cq] = G0[erow * MMA_LD + c0 + cq];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
                if (erow < n) {
                    a = *reinterpret_cast<const uint4*>(p.q + (row0 + erow * rs) * KD + c0 + 8 * u);
                    b = *reinterpret_cast<const uint4*>(p.k + (row0 + erow * rs) * KD + c0 + 8 * u);
                }
                float x[8], y[8];
                bf16x8(a, x);
                bf16x8(b, y);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q[8 * u + e] = x[e];
                    k[8 * u + e] = y[e];
                }
            }
            const float sq = scale * vNq[erow], sk = vNk[erow];
            float kh[16], kc[16];
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const float e = gq[cq] - vPiv[c0 + cq];
                const float ep = __expf(e), em = __expf(-e);
                kh[cq] = sk * k[cq] * ep;
                kc[cq] = sk * k[cq] * em;
                q[cq] = sq * q[cq] * ep;   // qh
            }
            float* gg = SG(G_G) + (size_t)erow * 128 + c0;
            float* gqh = SG(G_QH) + (size_t)erow * 128 + c0;
            float* gkh = SG(G_KH) + (size_t)erow * 128 + c0;
            float* gkc = SG(G_KC) + (size_t)erow * 128 + c0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                *reinterpret_cast<float4*>(gg + 4 * u) = make_float4(gq[4 * u], gq[4 * u + 1], gq[4 * u + 2], gq[4 * u + 3]);
                *reinterpret_cast<float4*>(gqh + 4 * u) = make_float4(q[4 * u], q[4 * u + 1], q[4 * u + 2], q[4 * u + 3]);
                *reinterpret_cast<float4*>(gkh + 4 * u) = make_float4(kh[4 * u], kh[4 * u + 1], kh[4 * u + 2], kh[4 * u + 3]);
                *reinterpret_cast<float4*>(gkc + 4 * u) = make_float4(kc[4 * u], kc[4 * u + 1], kc[4 * u + 2], kc[4 * u + 3]);
                st_km4(S1, erow, c0 + 4 * u, kh[4 * u], kh[4 * u + 1], kh[4 * u + 2], kh[4 * u + 3]);
                st_km4(S2, erow, c0 + 4 * u, kc[4 * u], kc[4 * u + 1], kc[4 * u + 2], kc[4 * u + 3]);
            }
        }
        __syncthreads();   // G in S0 read by all
        stage_km(S0, SG(G_QH), tid, [](int) { return 1.f; });   // G_QH rows were written by other threads:
        // the barrier above orders them (global writes visible within the CTA after __syncthreads)

        // ---- Aqk = tril(qh kc^T) -> ACC;  Pm = strict(kh kc^T) -> DKC ------------------------
        to_mma();
        if (tid == 0) {
            umma128(tmem + T_ACC, smem_u32(S0), smem_u32(S2), false);
            umma128(tmem + T_DKC, smem_u32(S1), smem_u32(S2), false);
        }
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq)
                if (32 * cs + cq > erow) x[cq] = 0.f;
            st_rowT32(SG(G_AQKT), erow, cs, x);
            tm_row(T_DKC, x);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq)
                if (32 * cs + cq >= erow) x[cq] = 0.f;
            st_row32(SG(G_PM), erow, cs, x);
            tc_fence_before();
            __syncthreads();   // S0 (qh) is free: the products that read it are done
            float* L = reinterpret_cast<float*>(S0);
            const float b = vBeta[erow];
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) {
                const int j = 32 * cs + cq;
                L[erow * MMA_LD + j] = (j == erow) ? 1.f : b * x[cq];
            }
        }
        __syncthreads();
        invert_unit_lower(reinterpret_cast<float*>(S0), warp, lane, tid);   // S0 = Li (padded)
        {
            const float* L = reinterpret_cast<const float*>(S0);
#pragma unroll 4
            for (int i = tid; i < 128 * 32; i += UM_THREADS) {
                const int r = i >> 5, c4 = (i & 31) * 4;
                *reinterpret_cast<float4*>(SG(G_LI) + r * 128 + c4) = *reinterpret_cast<const float4*>(L + r * MMA_LD + c4);
            }
        }
        // S2 = Sp^T (K-major: rows v, columns d): Sp^T[v][d] = e^{P_d} S0[d][v]
        stage_kmT(S2, Sc, warp, lane, [&](int r) { return __expf(vPiv[r]); });
        __syncthreads();   // Li spilled
        stage_km(S0, SG(G_LI), tid, [](int) { return 1.f; });   // S0 = Li (K-major)

        // ---- y0 = v - kh Sp -> ACC; y^T -> S1 ------------------------------------------------
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S1), smem_u32(S2), false);
        float vin[32];
        {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint4 a = make_uint4(0u, 0u, 0u, 0u);
                if (erow < n) a = *reinterpret_cast<const uint4*>(p.v + (row0 + erow * rs) * VD + 32 * cs + 8 * u);
                float x[8];
                bf16x8(a, x);
#pragma unroll
                for (int e = 0; e < 8; ++e) vin[8 * u + e] = x[e];
            }
        }
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) x[cq] = vin[cq] - x[cq];
            st_row32(SG(G_Y0), erow, cs, x);
            const float b = vBeta[erow];
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) x[cq] *= b;
            tc_fence_before();
            __syncthreads();   // S1 (kh) free
            km_rowT32(S1, erow, cs, x);   // y^T
        }
        // ---- rho = Li y -> ACC; rho -> S2 (K-major) and scratch ---------------------------
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S0), smem_u32(S1), false);
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
            st_row32(SG(G_RHO), erow, cs, x);
            km_row32(S2, erow, cs, x);   // S2 (Sp^T) free: its product is done
        }
        stage_km_bf16(S0, p.dout, row0, rs, n, tid);   // S0 = do (Li is in scratch)
        // ---- W = tril(do rho^T) -> ACC -----------------------------------------------------
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S0), smem_u32(S2), false);
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq)
                if (32 * cs + cq > erow) x[cq] = 0.f;
            st_row32(SG(G_W), erow, cs, x);
            st_rowT32(SG(G_WT), erow, cs, x);
        }
        __syncthreads();   // G_AQKT complete (written in an earlier epilogue)
        // ---- drho = Aqk^T do + kc Ze -> ACC ------------------------------------------------
        stage_km(S1, SG(G_AQKT), tid, [](int) { return 1.f; });       // A = Aqk^T  (rows s, columns t)
        stage_kmT_bf16(S2, p.dout, row0, rs, n, warp, lane);          // B = do^T   (rows v, columns t)
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S1), smem_u32(S2), false);
        commit_wait();
        tc_fence_before();
        __syncthreads();
        stage_km(S1, SG(G_KC), tid, [](int) { return 1.f; });         // A = kc     (rows s, columns d)
        {   // B = Ze^T (rows v, columns d): Ze^T[v][d] = e^{G_last,d - P_d} Z[d][v]; exit rowsum(Z * S0) on the way
            const int r = 32 * (warp >> 2) + lane, cb = warp & 3;
            float z[32], s0[32];
            ld_row32(Z, r, cb, z);
            ld_row32(Sc, r, cb, s0);
            float dot = 0.f;
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) dot = fmaf(z[cq], s0[cq], dot);
            vExR[cb * 128 + r] = dot;
            const float f = __expf(vTmp[r]);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) z[cq] *= f;
            km_rowT32(S2, r, cb, z);
        }
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S1), smem_u32(S2), true);
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
            tc_fence_before();
            __syncthreads();   // S1 free
            km_rowT32(S1, erow, cs, x);   // drho^T (rows v, columns s)
        }
        stage_kmT(S2, SG(G_LI), warp, lane, [](int) { return 1.f; });   // A = Li^T (rows t, columns s)
        // ---- dy = Li^T drho -> ACC;  dv = beta dy;  dbeta = rowsum(dy y0) ------------------
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S2), smem_u32(S1), false);
        float y0r[32];
        ld_row32(SG(G_Y0), erow, cs, y0r);
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
            const float b = vBeta[erow];
            float part = 0.f;
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) part = fmaf(x[cq], y0r[cq], part);
            vDbP[cs * 128 + erow] = part;
            if (erow < n) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<float4*>(p.dv + (row0 + erow * rs) * VD + 32 * cs + 4 * u) =
                        make_float4(b * x[4 * u], b * x[4 * u + 1], b * x[4 * u + 2], b * x[4 * u + 3]);
            }
            tc_fence_before();
            __syncthreads();   // S1 free
            km_row32(S1, erow, cs, x);   // dy (rows t, columns v)
        }
        stage_km(S2, SG(G_RHO), tid, [](int) { return 1.f; });
        // ---- X = strict(dy rho^T) -> ACC;  dbeta -= rowsum(X Pm) --------------------------
        to_mma();
        if (tid == 0) umma128(tmem + T_ACC, smem_u32(S1), smem_u32(S2), false);
        float pmr[32];
        ld_row32(SG(G_PM), erow, cs, pmr);
        commit_wait();
        {
            float x[32];
            tm_row(T_ACC, x);
            float part = 0.f;
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) {
                if (32 * cs + cq >= erow) x[cq] = 0.f;
                part = fmaf(-x[cq], pmr[cq], part);
            }
            vDbP[cs * 128 + erow] += part;
            st_row32(SG(G_X), erow, cs, x);
            st_rowT32(SG(G_XT), erow, cs, x);
        }
        tc_fence_before();
        __syncthreads();
        // ---- Sp -> S2: DKH = dy Sp^T, DQH = do Sp^T (S0 = do, S1 = dy) ---------------------
        stage_km(S2, Sc, tid, [&](int r) { return __expf(vPiv[r]); });
        to_mma();
        if (tid == 0) {
            umma128(tmem + T_DKH, smem_u32(S1), smem_u32(S2), false);
            umma128(tmem + T_DQH, smem_u32(S0), smem_u32(S2), false);
        }
        commit_wait();
        tc_fence_before();
        __syncthreads();
        // ---- DKC = rho Ze^T; exit colsum(kc * rho Ze^T) ------------------------------------
        stage_km(S0, SG(G_RHO), tid, [](int) { return 1.f; });
        stage_km(S1, Z, tid, [&](int r) { return __expf(vTmp[r]); });   // Ze (rows d, columns v)
        to_mma();
        if (tid == 0) umma128(tmem + T_DKC, smem_u32(S0), smem_u32(S1), false);
        float kcr[32];
        ld_row32(SG(G_KC), erow, cs, kcr);
        commit_wait();
        {
            float x[32];
            tm_row(T_DKC, x);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) x[cq] *= kcr[cq];
            const float colsum = warp_colsum32(x, lane);   // column 32 cs + lane over this warp's 32 rows
            vExC[qr * 128 + 32 * cs + lane] = colsum;
        }
        tc_fence_before();
        __syncthreads();
        // ---- DQH += W kc;  DKH += X kc  (B = kc^T: rows d, columns s) ------------------------
        stage_km(S0, SG(G_W), tid, [](int) { return 1.f; });
        stage_km(S1, SG(G_X), tid, [](int) { return 1.f; });
        stage_kmT(S2, SG(G_KC), warp, lane, [](int) { return 1.f; });
        to_mma();
        if (tid == 0) {
            umma128(tmem + T_DQH, smem_u32(S0), smem_u32(S2), true);
            umma128(tmem + T_DKH, smem_u32(S1), smem_u32(S2), true);
        }
        commit_wait();
        tc_fence_before();
        __syncthreads();
        // ---- DKC += W^T qh  (A = W^T: rows s, columns t; B = qh^T: rows d, columns t) --------
        stage_km(S0, SG(G_WT), tid, [](int) { return 1.f; });
        stage_kmT(S2, SG(G_QH), warp, lane, [](int) { return 1.f; });
        stage_km(S1, SG(G_XT), tid, [](int) { return 1.f; });        // for the next product
        to_mma();
        if (tid == 0) umma128(tmem + T_DKC, smem_u32(S0), smem_u32(S2), true);
        commit_wait();
        tc_fence_before();
        __syncthreads();
        // ---- DKC -= X^T (beta kh)  (B = -(beta kh)^T: rows d, columns t) ---------------------
        stage_kmT(S0, SG(G_KH), warp, lane, [&](int r) { return -vBeta[r]; });
        to_mma();
        if (tid == 0) umma128(tmem + T_DKC, smem_u32(S1), smem_u32(S0), true);
        commit_wait();

        // ---- outputs: dq, dk, dG (-> S2 padded), then dg by a reverse prefix sum ------------
        // (two 16-column halves of the thread's row segment)
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            const int c0 = 32 * cs + 16 * hf;
            float dqh[16], dkh[16], dkc[16], gq[16], q[16], k[16];
            tmem_ld16(trow + T_DQH + 16u * hf, dqh);
            tmem_ld16(trow + T_DKH + 16u * hf, dkh);
            tmem_ld16(trow + T_DKC + 16u * hf, dkc);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 gv = *reinterpret_cast<const float4*>(SG(G_G) + (size_t)erow * 128 + c0 + 4 * u);
                gq[4 * u] = gv.x; gq[4 * u + 1] = gv.y; gq[4 * u + 2] = gv.z; gq[4 * u + 3] = gv.w;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
                if (erow < n) {
                    a = *reinterpret_cast<const uint4*>(p.q + (row0 + erow * rs) * KD + c0 + 8 * u);
                    b = *reinterpret_cast<const uint4*>(p.k + (row0 + erow * rs) * KD + c0 + 8 * u);
                }
                float x[8], y[8];
                bf16x8(a, x);
                bf16x8(b, y);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q[8 * u + e] = x[e];
                    k[8 * u + e] = y[e];
                }
            }
            const float nb = -vBeta[erow], sq = scale * vNq[erow], sk = vNk[erow];
            float* DG = reinterpret_cast<float*>(S2);
            float oq[16], ok[16];
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const int j = c0 + cq;
                const float e = gq[cq] - vPiv[j];
                const float ep = __expf(e), em = __expf(-e);
                const float dkh_t = nb * dkh[cq];
                const float kk = sk * k[cq];
                DG[erow * MMA_LD + j] = sq * q[cq] * ep * dqh[cq] + kk * ep * dkh_t - kk * em * dkc[cq];
                oq[cq] = scale * dqh[cq] * ep;          // with the q/k norm: w.r.t. the normalised q, k
                ok[cq] = dkh_t * ep + dkc[cq] * em;
            }
            if (erow < n) {
                float* dq = p.dq + (row0 + erow * rs) * KD + c0;
                float* dk = p.dk + (row0 + erow * rs) * KD + c0;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    *reinterpret_cast<float4*>(dq + 4 * u) = make_float4(oq[4 * u], oq[4 * u + 1], oq[4 * u + 2], oq[4 * u + 3]);
                    *reinterpret_cast<float4*>(dk + 4 * u) = make_float4(ok[4 * u], ok[4 * u + 1], ok[4 * u + 2], ok[4 * u + 3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (tid < KD) {   // dg: reverse prefix sum over the valid rows, exit terms at row n - 1
            const float* DG = reinterpret_cast<const float*>(S2);
            float acc = __expf(vGl[tid]) * ((vExR[tid] + vExR[128 + tid]) + (vExR[256 + tid] + vExR[384 + tid])) +
                        ((vExC[tid] + vExC[128 + tid]) + (vExC[256 + tid] + vExC[384 + tid]));
            for (int r = n - 1; r >= 0; --r) {
                acc += DG[r * MMA_LD + tid];
                p.dg[(row0 + r * rs) * KD + tid] = acc;
            }
        }
        if (tid >= KD && tid < KD + BT && tid - KD < n) {
            const int r = tid - KD;
            p.dbeta[row0 + r * rs] = (vDbP[r] + vDbP[128 + r]) + (vDbP[256 + r] + vDbP[384 + r]);
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        if (*sFlag != 0) atomicOr(p.status, STATUS_TIMEOUT);
        // every product issued has completed before TMEM is freed (after the
        // last commit_wait the barrier's pending phase has parity `phase`)
        mma_commit(bar);
        mbar_wait(bar, phase, DRAIN_LIMIT);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, T_COLS);
}

cudaError_t launch_bwd_umma(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream) {
    if (fp.nslots == 0 || ctas == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)UM_SMEM);
    if (e != cudaSuccess) return e;
    kda_bwd_umma_kernel<<<ctas, UM_THREADS, UM_SMEM, stream>>>(p, fp);
    return cudaGetLastError();
}

}  // namespace kda
