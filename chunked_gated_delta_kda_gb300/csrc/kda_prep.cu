// Chunk-parallel half of the chunked KDA forward ("prep"): for one
// (chunk, head) it computes, from q, k, v, g, beta,
//   - the gate prefix sum G = cumsum(g) inside the chunk       (step M1)
//   - A  = beta_c * sum_d k_c k_i exp(G_c - G_i), i < c        (step M2)
//     A2 = sum_d (scale q_c) k_i exp(G_c - G_i),  i <= c        (M4's A2)
//   - (I + A)^-1 by blocked forward substitution               (step M2)
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
// Factoring.  With a pivot P (per dimension, the prefix sum at row 64),
//   E = exp(G - P),  F = exp(P - G),
//   Lk = k E, Lq = (scale q) E, R = k F,  so that A_raw = Lk R^T, A2_raw = Lq R^T.
// Two kernels of one template share everything after the gated products:
//   * fast (fp16 gated operands): when every Lk, Lq, R of the chunk fits
//     comfortably in fp16, the other operands are exact column / row
//     rescalings of these tiles and need no tiles of their own:
//       exp(G) k = Lk diag(exp(P))      ->  w = ((I+A)^-1 diag(beta) Lk) diag(exp(P))
//       kg       = R  diag(exp(G_last - P)) -> Nm = -diag(exp(G_last-P)) R^T w
//       qg       = Lq diag(exp(P))      ->  Qe = Lq diag(exp(P)) - A2 w
//     with beta folded into the columns of the inverse.
//   * wide (bf16 gated operands): chunks whose factors would overflow fp16
//     (strong decay inside the chunk) are queued by the fast kernel and
//     redone by this one, which builds exp(G) k, kg, qg and beta v as
//     separate fp16 tiles.  The fast kernel queues a chunk as soon as its
//     gate prefix alone shows a move from the pivot row that fp16 factors
//     cannot hold, before any fp16 gating, and otherwise after the exact
//     range check of its fp16 operands.  A chunk whose decay from the pivot
//     row exceeds the factor cap is flagged: its (sequence, head) is then
//     recomputed exactly, token by token, after the scan.
// Both kernels load a chunk's raw q, k, v tiles by tensor-map copies and
// compute the gate prefix with the same thread mapping; each has its own
// register allocation, so the wide code costs the fast kernel nothing.
//
// GB300 mapping.  Persistent kernels: one 512-thread CTA per SM walks the
// work items.  The 128-wide contractions run on tcgen05 tensor cores with
// fp16 operands (bf16 for the wide kernel's gated operands) and fp32
// accumulators in TMEM.  The prefix sum, the gated operands and the 16x16
// diagonal blocks of the inverse run on CUDA cores in fp32; the 16 -> 32 and
// 32 -> 64 merges of the inverse on warp-level TF32 tensor-core products
// (mma.sync, fp32 accumulation); the 64 -> 128 merge on tcgen05 with fp16
// operands.  While one chunk computes, its successor's input rows are
// prefetched into L2.
#include <cuda.h>            // CUtensorMap (types only; the encoder comes through the runtime)
#include <cudaTypedefs.h>
#include <mutex>

#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int PREP_THREADS = 512;
constexpr float LOG2E = 1.4426950408889634f;
// exp2 argument cap: 2^115 ~ e^80, the page's decay cap; keeps every factor
// finite so that a zero operand never meets an infinite one.
constexpr float EXP2_CAP = 115.0f;
// The fast kernel keeps a chunk only if every gated operand (Lk, Lq, R) is
// below this (fp16 max is 65504; the margin keeps products and sums finite).
// v is not checked: it is an fp16 operand in both kernels.
constexpr float FP16_SAFE = 16384.0f;

// Shared-memory regions (bytes from the 1024-aligned base).
//                  fast kernel (layout 0 | layout 1)          wide kernel (layout 0)
//   0    .. 64K :  raw k | raw v -> Lk | v16 -> w | u         raw k | raw v -> Lk | Lq -> qg | kg
//   64K  .. 96K :  raw q -> Lq    | R                         raw q -> R -> merge tiles -> Ainv
//                                                              -> Qe staging
//   96K  .. 128K:  R              | merge tiles -> Ainv       RHS (k part) -> w -> Nm staging
//   128K .. 160K:  merge tiles -> Ainv | raw q -> Lq          RHS (v part) -> u -> Bc staging
//   160K .. 208K:  fp32 diag blocks -> A2 (160K .. 192K)      qg stash -> fp32 diag blocks -> A2
//                  -> output staging 1; prefix totals at 192K -> Oi staging; prefix totals at 192K
// The fast kernel's chunks alternate between its two layouts, so that the
// next chunk's raw q (in place of this chunk's inverse, or of its R) and raw
// k, v (in place of w | u) can be loaded while this chunk's output tiles are
// staged in 96K .. 128K and 160K .. 192K.  The wide kernel keeps layout 0
// (raw q at 64K, requested once the Qe staging there has been stored); its
// gating reads each 16-byte piece of the raw tiles before it writes the same
// piece of any region, so the wide operands can be written over them.
constexpr uint32_t RM = 213248;            // misc
constexpr uint32_t M_G64 = RM;             // f32[128]  G at the pivot row (log2 units)
constexpr uint32_t M_GL = RM + 512;        // f32[128]  G at the last row (log2 units)
constexpr uint32_t M_BETA = RM + 1024;     // f32[128]
constexpr uint32_t M_INVQ = RM + 1536;     // f32[128]  scale / ||q|| (or scale)
constexpr uint32_t M_INVK = RM + 2048;     // f32[128]  1 / ||k|| (or 1)
constexpr uint32_t M_EP = RM + 2560;       // f32[128]  exp(P)
constexpr uint32_t M_CL = RM + 3072;       // f32[128]  exp(G_last - P), capped
constexpr uint32_t M_BAR = RM + 7680;      // mbarrier
constexpr uint32_t M_BAR2 = RM + 7688;     // mbarrier of the second transition product
constexpr uint32_t M_BARD = RM + 7696;     // mbarrier: every issued product done (before TMEM is freed)
constexpr uint32_t M_RAWB = RM + 7704;     // mbarrier: a chunk's raw q / k / v tiles landed
constexpr uint32_t M_TMEM = RM + 7744;     // TMEM base address
constexpr uint32_t M_FLAG = RM + 7748;     // failure flag
constexpr uint32_t SMEM_USED = RM + 7808;
constexpr uint32_t PREP_SMEM = SMEM_USED + 1024;  // + alignment slack

constexpr uint32_t RW = 163840;
// fp32 diagonal 64-blocks of (the strictly lower part of) A, then of its
// inverse, row stride 68 floats (conflict-free column walks).
constexpr int DS = 68;
constexpr uint32_t W_DIAG = RW;                          // 2 x 64 x 68 floats = 34816 B
constexpr uint32_t W_TMP = RW + 2 * 64 * DS * 4;         // merge temps, up to 10 KB
static_assert(W_TMP + 2 * 1280 * 4 <= RM, "merge temps overlap the misc block");
// the gate prefix-scan totals ([32 row groups][129] fp32), clear
// of the output staging buffers that may still be draining when they are written
constexpr uint32_t W_TOT = 196608;
static_assert(W_TOT + 32 * 129 * 4 <= RM, "prefix totals overlap the misc block");
// fast kernel: the two 32 KB staging buffers of the output tiles
constexpr uint32_t ST0 = 98304;
constexpr uint32_t ST1 = RW;
static_assert(PREP_SMEM <= 232448, "shared memory above the 227 KB limit");

// Fixed region map of the wide kernel (the fast kernel takes Lq, R and the
// inverse's region from its chunk's layout, and has Lk, the WY product's
// right-hand side and w | u at 0).
namespace wide_map {
constexpr uint32_t LQ = 32768;
constexpr uint32_t RR = 65536;     // R
constexpr uint32_t Y = 65536;      // merge tiles, then Ainv (over R)
constexpr uint32_t B2 = 98304;     // B operand of the WY product (N = 256): [beta exp(G) k | beta v]
constexpr uint32_t WU = 98304;     // w | u (N = 256), over B2
constexpr uint32_t KGT = 32768;    // kg: A operand (MN-major) of the Nm | Bc product, over Lq
constexpr uint32_t QS = 0;         // qg for the Qe epilogue, over Lk
// staging of the output tiles for the bulk stores: Qe and Oi once the first
// transition product is done (over Ainv and A2), Nm and Bc once the second
// is (over w | u)
constexpr uint32_t ST_QE = 65536;
constexpr uint32_t ST_OI = RW;
constexpr uint32_t ST_NM = 98304;
constexpr uint32_t ST_BC = 131072;
}  // namespace wide_map
// The fast kernel's gate-only check: a chunk whose gate prefix moves more
// than this (log2 units) between the pivot row and the chunk's first or last
// row in some dimension needs a factor above 2^18, which the fp16 range
// check passes only for |k| or |q| below 2^-4 there; such chunks are queued
// for the wide kernel without fp16 gating.
constexpr float WIDE_SPAN = 18.0f;

// max that propagates NaN (an operand 0 * inf must not pass the range check)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// Read-once input rows (one head's rows of one chunk): loaded with an L2
// evict-first policy so that they leave L2 ahead of the prefetched rows of
// the next chunk.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float4 ldg_ef_f4(const void* p, uint64_t pol) {
    float4 r;
    asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ void unpack8_bf16(const uint4 u, float (&x)[8]) {
    float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y; x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

// Warp-level tf32 tensor-core product D += A B (m16n8k8, fp32 accumulate),
// used for the small 16x16 / 32x32 merges of the inverse.  Fragments:
// g = lane / 4, t = lane % 4;  A: (g, t) (g+8, t) (g, t+4) (g+8, t+4);
// B: (k = t, n = g) (k = t+4, n = g);  D: (g, 2t) (g, 2t+1) (g+8, 2t) (g+8, 2t+1).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One 16 x 16 output tile of  C + A B  with A = rows [ar, ar+16) x cols
// [ac, ac+K) and B = rows [br, br+K) x cols [bc, bc+16) of fp32 matrices in
// shared memory (row strides sa, sb); C arrives and leaves in D-fragment
// layout, two 8-column halves.
template <int K>
__device__ __forceinline__ void mma_tile16(float (&c)[2][4], const float* A, int sa, const float* B, int sb,
                                           int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < K / 8; ++ks) {
        uint32_t a[4];
        a[0] = to_tf32(A[g * sa + ks * 8 + t]);
        a[1] = to_tf32(A[(g + 8) * sa + ks * 8 + t]);
        a[2] = to_tf32(A[g * sa + ks * 8 + t + 4]);
        a[3] = to_tf32(A[(g + 8) * sa + ks * 8 + t + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = to_tf32(B[(ks * 8 + t) * sb + nt * 8 + g]);
            const uint32_t b1 = to_tf32(B[(ks * 8 + t + 4) * sb + nt * 8 + g]);
            mma_tf32(c[nt], a, b0, b1);
        }
    }
}

// Load / store a 16 x 16 fp32 tile (row stride s) in D-fragment layout.
__device__ __forceinline__ void tile16_load(float (&c)[2][4], const float* M, int s, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        c[nt][0] = M[g * s + nt * 8 + 2 * t];
        c[nt][1] = M[g * s + nt * 8 + 2 * t + 1];
        c[nt][2] = M[(g + 8) * s + nt * 8 + 2 * t];
        c[nt][3] = M[(g + 8) * s + nt * 8 + 2 * t + 1];
    }
}
__device__ __forceinline__ void tile16_store(const float (&c)[2][4], float* M, int s, int lane, float sign) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        M[g * s + nt * 8 + 2 * t] = sign * c[nt][0];
        M[g * s + nt * 8 + 2 * t + 1] = sign * c[nt][1];
        M[(g + 8) * s + nt * 8 + 2 * t] = sign * c[nt][2];
        M[(g + 8) * s + nt * 8 + 2 * t + 1] = sign * c[nt][3];
    }
}

// 128B-swizzled tile operand: K-major (rows = M or N, 128 B of K per row,
// 64-wide K slabs `rows` rows apart) or MN-major (rows = K, 64-wide MN atoms
// one slab apart).
struct Operand {
    uint32_t base;
    bool mn_major;
    uint32_t rows;
};

__device__ __forceinline__ uint64_t op_desc(const Operand& o, int ks) {
    if (o.mn_major) return smem_desc(o.base + (uint32_t)ks * 2048u, o.rows * 128u, 1024u, SW_128B);
    return smem_desc(o.base + (uint32_t)(ks >> 2) * o.rows * 128u + (uint32_t)(ks & 3) * 32u, 16u, 1024u,
                     SW_128B);
}

// Descriptor advance per k-step, in the 16-byte units of the start-address
// field (adding it to a base descriptor never carries out of the field:
// shared addresses stay below 256 KB).
__device__ __forceinline__ uint64_t op_step(const Operand& o, int ks) {
    if (o.mn_major) return (uint64_t)ks * 128u;
    return (uint64_t)((ks >> 2) * (int)o.rows * 8 + (ks & 3) * 2);
}

__device__ __forceinline__ void mma_128(uint32_t d_tmem, const Operand& a, const Operand& b, uint32_t idesc,
                                        int ksteps) {
    const uint64_t da = op_desc(a, 0), db = op_desc(b, 0);
#pragma unroll
    for (int ks = 0; ks < ksteps; ++ks) mma_f16(d_tmem, da + op_step(a, ks), db + op_step(b, ks), idesc, ks > 0);
}

__device__ __forceinline__ void bar_sync_named(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier between a phase's shared-memory / TMEM writes and the tensor core
// reading them (or a new MMA overwriting TMEM that was read).
__device__ __forceinline__ void sync_for_mma() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}


__device__ __forceinline__ void prefetch_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// L2 prefetch of one chunk's input rows (q, k, v, g): one row per thread,
// one 128-byte line per instruction.  Plain line prefetches go through the
// load path; bulk prefetches would queue behind the previous tile's bulk
// stores and stall the issuing threads.
__device__ __forceinline__ void prefetch_chunk(const FwdParams& p, const ChunkRef& c, int h, int tid) {
    const int t = tid & 127;
    if (t >= c.len) return;
    const size_t row = (size_t)(c.tok0 + t) * p.H + h;
    switch (tid >> 7) {
        case 0:
            prefetch_line(p.beta + row);
            prefetch_line(p.q + row * KD);
            prefetch_line(p.q + row * KD + 64);
            break;
        case 1:
            prefetch_line(p.k + row * KD);
            prefetch_line(p.k + row * KD + 64);
            break;
        case 2:
            prefetch_line(p.v + row * VD);
            prefetch_line(p.v + row * VD + 64);
            break;
        default:
            prefetch_line(p.g + row * KD);
            prefetch_line(p.g + row * KD + 32);
            prefetch_line(p.g + row * KD + 64);
            prefetch_line(p.g + row * KD + 96);
            break;
    }
}

// Work iteration.  Fast kernel: every (slot, head) item, grid-stride,
// skipping empty slots.  Wide kernel: the entries of the queue the fast
// kernel filled.
template <bool FAST>
__device__ __forceinline__ bool fetch_item(const FwdParams& p, long long& idx, long long& item, ChunkRef& c,
                                           int& h) {
    if (FAST) {
        // 32-bit index arithmetic (nslots * H < 2^31, checked on the host)
        const uint32_t nitems = (uint32_t)p.nslots * (uint32_t)p.H;
        while (idx < (long long)nitems) {
            const uint32_t ui = (uint32_t)idx, slot = ui / (uint32_t)p.H;
            if (slot_chunk(p, (int)slot, c)) {
                item = idx;
                h = (int)(ui - slot * (uint32_t)p.H);
                return true;
            }
            idx += gridDim.x;
        }
        return false;
    } else {
        const long long n = (long long)*reinterpret_cast<volatile uint32_t*>(p.wide_count);
        while (idx < n) {
            item = p.wide_list[idx];
            if (slot_chunk(p, (int)(item / p.H), c)) {
                h = (int)(item % p.H);
                return true;
            }
            idx += gridDim.x;
        }
        return false;
    }
}

// Wide-kernel gating of one thread's 4 rows x 8 dimensions (G: the gate
// prefix minus the pivot, log2 units).  Lk, Lq, R bf16
// (capped factors) over the raw tiles; RHS = [beta exp(G) k | beta v] fp16
// and qg fp16 in their own regions; kg fp16 parked in tensor memory columns
// 256 .. 319 (free until the WY product), 16 per warp of a lane quarter,
// until the region of Lq is free.  exp(G) = E exp(P) <= 1.
template <bool L2NORM>
__device__ __forceinline__ void wide_gating(uint8_t* sm, const float (&G)[4][8], int tg0, int d8, int len,
                                            uint32_t oRawQ, uint32_t kg_col) {
    const float* sBeta = reinterpret_cast<const float*>(sm + M_BETA);
    const float* sInvQ = reinterpret_cast<const float*>(sm + M_INVQ);
    const float* sInvK = reinterpret_cast<const float*>(sm + M_INVK);
    const float* sEP = reinterpret_cast<const float*>(sm + M_EP);
    const float* sCL = reinterpret_cast<const float*>(sm + M_CL);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = tg0 + r;
        const uint32_t off = sw128_off(t, d8, 128);
        uint4 kc = *reinterpret_cast<const uint4*>(sm + off);
        uint4 vc = *reinterpret_cast<const uint4*>(sm + 32768 + off);
        uint4 qc = *reinterpret_cast<const uint4*>(sm + oRawQ + off);
        if (len < BT && t >= len) kc = vc = qc = make_uint4(0u, 0u, 0u, 0u);   // tail chunks only
        float kf[8], qf[8], vf[8];
        unpack8_bf16(kc, kf);
        unpack8_bf16(qc, qf);
        unpack8_bf16(vc, vf);
        const float ik = L2NORM ? sInvK[t] : 1.f, iq = sInvQ[t], b = sBeta[t];
        uint32_t lk[4], lqv[4], rk[4], bk[4], bv[4], qg[4], kg[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const float g0 = G[r][j], g1 = G[r][j + 1];
            const float E0 = ex2(fminf(g0, EXP2_CAP)), E1 = ex2(fminf(g1, EXP2_CAP));
            const float F0 = ex2(fminf(-g0, EXP2_CAP)), F1 = ex2(fminf(-g1, EXP2_CAP));
            const float k0 = kf[j] * ik, k1 = kf[j + 1] * ik;
            const float q0 = qf[j] * iq, q1 = qf[j + 1] * iq;
            const float eg0 = E0 * sEP[d8 + j], eg1 = E1 * sEP[d8 + j + 1];
            lk[j / 2] = pack_bf16(k0 * E0, k1 * E1);
            lqv[j / 2] = pack_bf16(q0 * E0, q1 * E1);
            rk[j / 2] = pack_bf16(k0 * F0, k1 * F1);
            bk[j / 2] = pack_f16(b * k0 * eg0, b * k1 * eg1);
            bv[j / 2] = pack_f16(b * vf[j], b * vf[j + 1]);
            qg[j / 2] = pack_f16(q0 * eg0, q1 * eg1);
            kg[j / 2] = pack_f16(k0 * F0 * sCL[d8 + j], k1 * F1 * sCL[d8 + j + 1]);
        }
        // every raw piece of this row was read above: its own pieces of the
        // regions below may now be overwritten
        sts_v4(sm, off, lk[0], lk[1], lk[2], lk[3]);
        sts_v4(sm, wide_map::LQ + off, lqv[0], lqv[1], lqv[2], lqv[3]);
        sts_v4(sm, wide_map::RR + off, rk[0], rk[1], rk[2], rk[3]);
        sts_v4(sm, wide_map::B2 + off, bk[0], bk[1], bk[2], bk[3]);
        sts_v4(sm, wide_map::B2 + 32768u + off, bv[0], bv[1], bv[2], bv[3]);
        sts_v4(sm, RW + off, qg[0], qg[1], qg[2], qg[3]);
        tmem_st4(kg_col + (uint32_t)(4 * r), kg[0], kg[1], kg[2], kg[3]);
    }
}

}  // namespace

template <bool L2NORM, bool FAST>
__global__ void __launch_bounds__(PREP_THREADS, 1)
    kda_prep_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int H = p.H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int lq = warp & 3;              // TMEM lane quarter of this warp
    const int cg = warp >> 2;             // column group (0..3) for TMEM read-backs
    const uint32_t lane_off = (uint32_t)(lq * 32) << 16;
    const int trow = lq * 32 + lane;      // TMEM lane = matrix row of this thread
    // thread 0 issues (and waits for) every bulk tile store and tensor load
    const bool bulk_thread = tid == 0;

    float* sG64 = reinterpret_cast<float*>(sm + M_G64);
    float* sGL = reinterpret_cast<float*>(sm + M_GL);
    float* sBeta = reinterpret_cast<float*>(sm + M_BETA);
    float* sInvQ = reinterpret_cast<float*>(sm + M_INVQ);
    float* sInvK = reinterpret_cast<float*>(sm + M_INVK);
    float* sEP = reinterpret_cast<float*>(sm + M_EP);
    float* sCL = reinterpret_cast<float*>(sm + M_CL);
    float* Wd = reinterpret_cast<float*>(sm + W_DIAG);
    float* Wt = reinterpret_cast<float*>(sm + W_TMP);
    const uint32_t bar = sbase + M_BAR;
    const uint32_t bar2 = sbase + M_BAR2;
    uint32_t phase2 = 0;
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(sm + M_FLAG);
    uint32_t phase = 0;

    long long idx = blockIdx.x, item = 0;
    ChunkRef c;
    int h = 0;
    bool have = fetch_item<FAST>(p, idx, item, c, h);
    if (!have) return;                    // uniform: nothing for this CTA

    if (warp == 0) {
        tmem_alloc(sbase + M_TMEM, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar2, 1);
        mbar_init(sbase + M_BARD, 1);
        mbar_init(sbase + M_RAWB, 1);
        fence_mbar_init();
        *sFlag = 0;
    }
    prefetch_chunk(p, c, h, tid);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + M_TMEM);

    // A chunk's raw k, v and q tiles arrive by tensor-map loads (128-byte
    // swizzled, the layout of the MMA operands) straight into the regions
    // where the gated operands are then computed in place (fast kernel: k -> Lk,
    // v -> the fp16 copy of v, q -> Lq).  Consecutive chunks of a CTA alternate
    // between two region layouts so that the next chunk's loads can be issued
    // while this chunk's output tiles are still being staged (layout 0 / 1:
    // Lq at 64K / 128K, R at 96K / 64K, the inverse at 128K / 96K).
    const uint32_t rawbar = sbase + M_RAWB;
    uint32_t rphase = 0;
    bool raw_pending = false;   // a raw load was issued and not yet waited for
    auto issue_raw = [&](const ChunkRef& cc, int hh, int lay_n) {   // thread 0
        const uint32_t qo = lay_n ? 131072u : 65536u;
        mbar_arrive_expect_tx(rawbar, 3u * 32768u);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(sbase + (uint32_t)half * 16384u, &tm_k, half * 64, hh, (int)cc.tok0, rawbar);
            tma_load_3d(sbase + 32768u + (uint32_t)half * 16384u, &tm_v, half * 64, hh, (int)cc.tok0, rawbar);
            tma_load_3d(sbase + qo + (uint32_t)half * 16384u, &tm_q, half * 64, hh, (int)cc.tok0, rawbar);
        }
    };
    int lay = 0;
    if (tid == 0) issue_raw(c, h, 0);
    raw_pending = true;

    // Bounded waits: once one has run out (flag set), later ones of this CTA
    // return at once, the item finishes on whatever the tensor memory holds
    // (its tiles are garbage; the status word reports the failure) and the
    // loop ends after it.  The flag is only set before the item's last CTA
    // barrier, so every thread sees the same value at the loop test.
    const uint32_t wlim = wait_limit_of(p);
    auto bounded_wait = [&](uint32_t b, uint32_t parity) {
        if (*sFlag == 0 && !mbar_wait(b, parity, wlim)) *sFlag = 1;
    };
    auto wait_mma = [&]() {
        bounded_wait(bar, phase);
        phase ^= 1;
        tc_fence_after();
    };
    // a chunk's raw tiles have landed; after a wait that ran out the load
    // stays pending and is drained before the CTA exits
    auto wait_raw = [&]() {
        bounded_wait(rawbar, rphase);
        if (*sFlag == 0) {
            rphase ^= 1;
            raw_pending = false;
        }
    };


    // a chunk's beta and gate rows are loaded into registers during the
    // previous chunk's epilogue
    const uint64_t efp = evict_first_policy();
    float4 gpre[4][2];
    float bpre = 0.f;
    auto load_g = [&](const ChunkRef& cc, int hh, int r) {
        const int d8 = (tid & 15) * 8;
        const int t = (tid >> 4) * 4 + r;
        gpre[r][0] = gpre[r][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < cc.len) {
            const size_t off = ((size_t)cc.tok0 * H + hh + (size_t)t * H) * KD + d8;
            gpre[r][0] = ldg_ef_f4(p.g + off, efp);
            gpre[r][1] = ldg_ef_f4(p.g + off + 4, efp);
        }
    };
    auto load_beta = [&](const ChunkRef& cc, int hh) {
        const size_t r0 = (size_t)cc.tok0 * H + hh;
        bpre = (tid < BT && tid < cc.len) ? __ldg(p.beta + r0 + (size_t)tid * H) : 0.f;
    };
    auto load_rows = [&](const ChunkRef& cc, int hh) {
#pragma unroll
        for (int r = 0; r < 4; ++r) load_g(cc, hh, r);
        load_beta(cc, hh);
    };
    ChunkRef none{};   // zero rows: loads nothing, defines the registers
    none.len = 0;
    load_rows(c, h);

    while (have && *sFlag == 0) {
        long long nidx = idx + gridDim.x, nitem = 0;
        ChunkRef cn;
        int hn = 0;
        const bool have_n = fetch_item<FAST>(p, nidx, nitem, cn, hn);
        const int len = c.len;
        const size_t row0 = (size_t)c.tok0 * H + h;
        // region offsets of this chunk's alternating layout (the raw q tile
        // lands at oRawQ in both kernels; the wide kernel's other regions are
        // fixed)
        const uint32_t oRawQ = lay ? 131072u : 65536u;   // fast kernel: Lq
        const uint32_t oRf = lay ? 65536u : 98304u;       // fast kernel: R

        // ------------------------------------------------------------------
        // Per-row scalars: beta, and the q / k scalings (scale, optional
        // L2 normalisation x / sqrt(sum x^2 + 1e-6)).
        // ------------------------------------------------------------------
        if (tid < BT) {
            sBeta[tid] = bpre;
            if (!L2NORM) {
                sInvQ[tid] = p.scale;
                sInvK[tid] = 1.f;
            }
        }
        if (L2NORM) {
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

        // ------------------------------------------------------------------
        // Phase 1: gate prefix sum (log2 units), pivot row 64, gated operands.
        // thread = 8 consecutive dimensions x 4 consecutive rows
        // ------------------------------------------------------------------
        const int d8 = (tid & 15) * 8;
        const int grp = tid >> 4;
        const int tg0 = grp * 4;
        float G[4][8];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 ga = gpre[r][0], gb = gpre[r][1];
            G[r][0] = ga.x; G[r][1] = ga.y; G[r][2] = ga.z; G[r][3] = ga.w;
            G[r][4] = gb.x; G[r][5] = gb.y; G[r][6] = gb.z; G[r][7] = gb.w;
        }
        float span = 0.f;   // fast kernel: the gate's move from the pivot row
        // [32 groups][129]: the odd row stride keeps the column-wise
        // prefix scan free of shared-memory bank conflicts
        constexpr int TS = 129;
        float* tot = reinterpret_cast<float*>(sm + W_TOT);
        {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[j] = fmaf(G[r][j], LOG2E, acc[j]);
                    G[r][j] = acc[j];
                }
#pragma unroll
            for (int j = 0; j < 8; ++j) tot[grp * TS + d8 + j] = acc[j];
        }
        __syncthreads();
        {   // exclusive prefix over the 32 row groups, four threads per
            // dimension: thread (d = tid / 4, quarter qq = tid % 4) scans
            // groups 8 qq .. 8 qq + 7 in order, then adds the totals of
            // the lower quarters (two shuffle steps among its 4 lanes)
            const int d = tid >> 2, qq = tid & 3;
            float v[8], run = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = tot[(8 * qq + i) * TS + d];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = v[i];
                v[i] = run;
                run += x;
            }
            float incl = run;
#pragma unroll
            for (int s2 = 1; s2 < 4; s2 <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, s2, 4);
                if (qq >= s2) incl += y;
            }
            const float base = incl - run;
#pragma unroll
            for (int i = 0; i < 8; ++i) tot[(8 * qq + i) * TS + d] = base + v[i];
            if (FAST) {   // the gate prefix at rows 63 and 127 (quarter totals)
                const float g63 = __shfl_sync(0xffffffffu, incl, 1, 4);
                const float g127 = __shfl_sync(0xffffffffu, incl, 3, 4);
                span = fmax_nan(fabsf(g63), fabsf(g127 - g63));
            }
        }
        // Fast kernel: the gate-only check, on this barrier.  A chunk whose
        // gate prefix moves plainly beyond what fp16 factors hold between
        // the pivot row (taken as row 63 here) and the chunk's first or last
        // row is queued for the wide kernel without fp16 gating.
        bool handoff_gate = false;
        if constexpr (FAST)
            handoff_gate = __syncthreads_or(!(span <= WIDE_SPAN)) != 0;
        else
            __syncthreads();
        {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float o = tot[grp * TS + d8 + j];
#pragma unroll
                for (int r = 0; r < 4; ++r) G[r][j] += o;
            }
            if (grp == 16) {
#pragma unroll
                for (int j = 0; j < 8; ++j) sG64[d8 + j] = G[0][j];
            }
            if (grp == 31) {
#pragma unroll
                for (int j = 0; j < 8; ++j) sGL[d8 + j] = G[3][j];
            }
        }
        if (bulk_thread) bulk_wait_read0();   // previous tile's bulk stores have read their staging
        __syncthreads();
        if (tid < 128) {
            const float P = sG64[tid];
            sEP[tid] = ex2(P);
            sCL[tid] = ex2(fminf(sGL[tid] - P, EXP2_CAP));
        }
        // only G - P is needed from here on: fold the pivot in once
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float P = sG64[d8 + j];
#pragma unroll
            for (int r = 0; r < 4; ++r) G[r][j] -= P;
        }
        bool handoff = handoff_gate;   // fast kernel: the chunk goes to the wide kernel's queue
        if constexpr (!FAST) __syncthreads();   // sEP / sCL are written
        // this chunk's raw k, v, q tiles have landed (rows past the
        // sequence's end hold other tokens or zeros: read as zero)
        wait_raw();
        if (FAST && !handoff) {
            float m = 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = tg0 + r;
                const uint32_t off = sw128_off(t, d8, 128);
                uint4 kc = *reinterpret_cast<const uint4*>(sm + off);
                uint4 vc = *reinterpret_cast<const uint4*>(sm + 32768 + off);
                uint4 qc = *reinterpret_cast<const uint4*>(sm + oRawQ + off);
                if (len < BT && t >= len) kc = vc = qc = make_uint4(0u, 0u, 0u, 0u);   // tail chunks only
                float kf[8], qf[8], vf[8];
                unpack8_bf16(kc, kf);
                unpack8_bf16(qc, qf);
                unpack8_bf16(vc, vf);
                const float ik = L2NORM ? sInvK[t] : 1.f, iq = sInvQ[t];
                uint32_t lk[4], lqv[4], rk[4], v16[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    // uncapped: a factor that overflows makes an operand
                    // infinite, which the range check sends to the wide kernel
                    const float E0 = ex2(G[r][j]), E1 = ex2(G[r][j + 1]);
                    const float F0 = ex2(-G[r][j]), F1 = ex2(-G[r][j + 1]);
                    const float k0 = kf[j] * ik, k1 = kf[j + 1] * ik;
                    const float q0 = qf[j] * iq, q1 = qf[j + 1] * iq;
                    const float a0 = k0 * E0, a1 = k1 * E1, b0 = q0 * E0, b1 = q1 * E1, c0 = k0 * F0, c1 = k1 * F1;
                    m = fmax_nan(m, fmax_nan(fmax_nan(fabsf(a0), fabsf(a1)), fmax_nan(fabsf(b0), fabsf(b1))));
                    m = fmax_nan(m, fmax_nan(fabsf(c0), fabsf(c1)));
                    lk[j / 2] = pack_f16(a0, a1);
                    lqv[j / 2] = pack_f16(b0, b1);
                    rk[j / 2] = pack_f16(c0, c1);
                    v16[j / 2] = pack_f16(vf[j], vf[j + 1]);
                }
                // in place over the raw tiles (each thread rewrites the 16
                // bytes it read), R into its own region
                sts_v4(sm, off, lk[0], lk[1], lk[2], lk[3]);
                sts_v4(sm, 32768 + off, v16[0], v16[1], v16[2], v16[3]);
                sts_v4(sm, oRawQ + off, lqv[0], lqv[1], lqv[2], lqv[3]);
                sts_v4(sm, oRf + off, rk[0], rk[1], rk[2], rk[3]);
            }
            // the range check; the same barrier hands the operands to the
            // tensor core
            fence_async_smem();
            tc_fence_before();
            handoff = __syncthreads_or(!(m <= FP16_SAFE)) != 0;
            tc_fence_after();
        }
        if constexpr (!FAST) {
            // beyond |G - P| = EXP2_CAP the capped factors no longer multiply
            // back to exp(G_c - G_i): this (sequence, head) is recomputed
            // token by token after the scan
            bool far = false;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int j = 0; j < 8; ++j) far = far || fabsf(G[r][j]) > EXP2_CAP;
            if (__any_sync(0xffffffffu, far) && lane == 0) p.exact_flags[(size_t)c.n * H + h] = 1u;
            wide_gating<L2NORM>(sm, G, tg0, d8, len, oRawQ, tmem + lane_off + 256u + (uint32_t)(cg * 16));
            tmem_st_wait();
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (handoff) {
            if (tid == 0) {
                const uint32_t slot_i = atomicAdd(p.wide_count, 1u);
                p.wide_list[slot_i] = (int32_t)item;
                // the next chunk's raw tiles go to regions this chunk no
                // longer needs (its operands, if any, are dropped)
                if (have_n) issue_raw(cn, hn, lay ^ 1);
            }
            if (have_n) raw_pending = true;
            if (have_n) prefetch_chunk(p, cn, hn, tid);
            load_rows(have_n ? cn : none, hn);
            __syncthreads();
        } else {
            if (tid == 0) {
                const uint32_t id = idesc_f16(FAST ? T_F16 : T_BF16, 128, 128, false, false);
                const Operand Lk{sbase, false, 128}, Lq{sbase + (FAST ? oRawQ : wide_map::LQ), false, 128},
                    R{sbase + (FAST ? oRf : wide_map::RR), false, 128};
                mma_128(tmem + 0, Lk, R, id, 8);     // A_raw  -> cols [0,128)
                mma_128(tmem + 128, Lq, R, id, 8);   // A2_raw -> cols [128,256)
                mma_commit(bar);
            }
            // the next chunk's rows stream into L2 while this one computes
            if (have_n) prefetch_chunk(p, cn, hn, tid);
            wait_mma();

            // the inverse's region (merge tiles, then Ainv)
            const uint32_t oY = FAST ? (lay ? 98304u : 131072u) : wide_map::Y;
            // --------------------------------------------------------------
            // Phase 2: A (strictly lower, times beta_row) from TMEM: diagonal
            // 64-blocks to fp32 (W), A10 to fp16 (YA).  The wide kernel first
            // moves kg and qg into regions 0 .. 64K (Lk and Lq are free).
            // --------------------------------------------------------------
            if constexpr (!FAST) {
                {
                    float kf[16];
                    tmem_ld16(tmem + lane_off + 256u + (uint32_t)(cg * 16), kf);
                    tmem_ld_wait();
                    const uint32_t* kg = reinterpret_cast<const uint32_t*>(kf);
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        sts_v4(sm, wide_map::KGT + sw128_off((tid >> 4) * 4 + r, (tid & 15) * 8, 128), kg[4 * r], kg[4 * r + 1], kg[4 * r + 2],
                               kg[4 * r + 3]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = (uint32_t)(tid + i * PREP_THREADS) * 16u;
                    *reinterpret_cast<uint4*>(sm + wide_map::QS + off) = *reinterpret_cast<const uint4*>(sm + RW + off);
                }
                __syncthreads();
            }
            {
                const int col0 = cg * 32;
                // warps whose block lies above the diagonal (row < 64, col >= 64) skip
                if (!(trow < 64 && col0 >= 64)) {
                    float x[32];
                    if (lq < cg) {            // above the diagonal (inside a 64-block): zeros
#pragma unroll
                        for (int j = 0; j < 32; ++j) x[j] = 0.f;
                    } else {
                        tmem_ld32(tmem + lane_off + (uint32_t)col0, x);
                        tmem_ld_wait();
                        const float b = sBeta[trow];
                        if (lq > cg) {        // below the diagonal: no mask needed
#pragma unroll
                            for (int j = 0; j < 32; ++j) x[j] *= b;
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) x[j] = (col0 + j < trow) ? b * x[j] : 0.f;
                        }
                    }
                    if (trow >= 64 && col0 < 64) {
#pragma unroll
                        for (int j = 0; j < 32; j += 8)
                            sts_v4(sm, oY + sw128_off(trow - 64, col0 + j, 64), pack_f16(x[j], x[j + 1]),
                                   pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]),
                                   pack_f16(x[j + 6], x[j + 7]));
                    } else {
                        float* dst = Wd + (trow >> 6) * 64 * DS + (trow & 63) * DS + (col0 & 63);
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();

            // --------------------------------------------------------------
            // Phase 3: (I + A)^-1.
            // Level 0: the eight 16x16 diagonal blocks, one column per
            // thread, forward substitution (unit diagonal implied; stored
            // parts are strictly lower, zeros elsewhere).
            // --------------------------------------------------------------
            {
                float x[16];
                const int blk = (tid >> 4) & 7, j = tid & 15;
                float* A0 = Wd + (blk >> 2) * 64 * DS + (blk & 3) * 16 * (DS + 1);
                if (tid < 128) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float s = 0.f;
#pragma unroll
                        for (int mm = 0; mm < i; ++mm) s = fmaf(A0[i * DS + mm], x[mm], s);
                        x[i] = (i == j) ? 1.f : (i < j ? 0.f : -s);
                    }
                }
                __syncthreads();
                if (tid < 128) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i > j) A0[i * DS + j] = x[i];
                }
                __syncthreads();
            }
            // Levels 1 and 2 inside each diagonal 64-block:
            //   inv([[X, 0], [Y, Z]]) = [[Xi, 0], [-Zi Y Xi, Zi]]
            // T = Y Xi = Y + Y Xs (Xs: stored strictly-lower part of Xi) into
            // a temp, then -Zi T = -(T + Zs T) in place of Y.  Products on
            // the tensor cores (warp-level tf32, fp32 accumulate).
            if (warp < 4) {
                // level 1: 4 merges of 16-blocks (2 per diagonal block), one warp each
                const int db = warp >> 1;
                const int C0 = (warp & 1) * 32, R0 = C0 + 16;
                float* Db = Wd + db * 64 * DS;
                float* T1 = Wt + warp * 384;   // 16 x 16, row stride 24 (conflict-free fragment loads)
                float acc[2][4];
                tile16_load(acc, Db + R0 * DS + C0, DS, lane);                           // Y
                mma_tile16<16>(acc, Db + R0 * DS + C0, DS, Db + C0 * DS + C0, DS, lane);  // + Y Xs
                tile16_store(acc, T1, 24, lane, 1.f);
                __syncwarp();
                mma_tile16<16>(acc, Db + R0 * DS + R0, DS, T1, 24, lane);               // T + Zs T
                tile16_store(acc, Db + R0 * DS + C0, DS, lane, -1.f);
            }
            __syncthreads();
            if (warp < 8) {
                // level 2: 2 merges of 32-blocks (one per diagonal block), one
                // 16x16 quadrant of the 32x32 result per warp
                const int db = warp >> 2;
                const int mr = ((warp >> 1) & 1) * 16, nc = (warp & 1) * 16;
                float* Db = Wd + db * 64 * DS;
                float* T2 = Wt + db * 1280;     // 32 x 32, row stride 40 (conflict-free fragment loads)
                float acc[2][4];
                tile16_load(acc, Db + (32 + mr) * DS + nc, DS, lane);                        // Y
                mma_tile16<32>(acc, Db + (32 + mr) * DS, DS, Db + nc, DS, lane);             // + Y Xs
                tile16_store(acc, T2 + mr * 40 + nc, 40, lane, 1.f);
                bar_sync_named(1, 256);
                mma_tile16<32>(acc, Db + (32 + mr) * DS + 32, DS, T2 + nc, 40, lane);        // T + Zs T
                tile16_store(acc, Db + (32 + mr) * DS + nc, DS, lane, -1.f);
            }
            __syncthreads();
            // Level 3 on tensor cores: L = -Q (A10 P), P / Q the inverses of
            // the two diagonal 64-blocks.  fp16 tiles: A10 [r][m] K-major
            // (written in phase 2; rows 64..127 of the M=128 MMA read the
            // next tile and land in TMEM lanes never read), P [m][c]
            // MN-major, Q [r'][r] K-major, T [r][c] MN-major.
            for (int e = tid; e < 64 * 32; e += PREP_THREADS) {
                const int r = e >> 5, c2 = (e & 31) * 2;
                const float* Pp = Wd + r * DS + c2;
                const float* Qp = Wd + 64 * DS + r * DS + c2;
                sts_u32(sm, oY + 8192u + sw128_off(r, c2, 64),
                        pack_f16(Pp[0] + (r == c2 ? 1.f : 0.f), Pp[1] + (r == c2 + 1 ? 1.f : 0.f)));
                sts_u32(sm, oY + 16384u + sw128_off(r, c2, 64),
                        pack_f16(Qp[0] + (r == c2 ? 1.f : 0.f), Qp[1] + (r == c2 + 1 ? 1.f : 0.f)));
            }
            sync_for_mma();
            if (tid == 0) {
                const Operand A10{sbase + oY, false, 64}, Ph{sbase + oY + 8192u, true, 64};
                mma_128(tmem + 0, A10, Ph, idesc_f16(T_F16, 128, 64, false, true), 4);   // T -> cols [0,64)
                mma_commit(bar);
            }
            wait_mma();
            if (lq < 2) {
                float x[16];
                tmem_ld16(tmem + lane_off + (uint32_t)(cg * 16), x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; j += 8)
                    sts_v4(sm, W_TMP + sw128_off(trow, cg * 16 + j, 64), pack_f16(x[j], x[j + 1]),
                           pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
            }
            sync_for_mma();
            if (tid == 0) {
                const Operand Qh{sbase + oY + 16384u, false, 64}, Th{sbase + W_TMP, true, 64};
                mma_128(tmem + 64, Qh, Th, idesc_f16(T_F16, 128, 64, false, true, /*neg_a=*/true), 4);  // L
                mma_commit(bar);
            }
            // Assemble (I + A)^-1 as fp16, K-major [c][i], in region Y:
            //   rows 0..63:  [P | 0],   rows 64..127: [L | Q]   (unit diagonal)
            // The fast kernel folds diag(beta) into its columns.  P (over A10,
            // read by the finished first merge product) and Q (over nothing)
            // are written while the second product runs; the zeros (over its
            // Q operand) and L (its result) after it.
            auto ainv_part = [&](int r, int c0) {
                float x[8];
                const float* src = Wd + (r >> 6) * 64 * DS + (r & 63) * DS + (c0 & 63);
                const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x[e] += (c0 + e == r) ? 1.f : 0.f;
                    if (FAST) x[e] *= sBeta[c0 + e];
                }
                sts_v4(sm, oY + sw128_off(r, c0, 128), pack_f16(x[0], x[1]), pack_f16(x[2], x[3]),
                       pack_f16(x[4], x[5]), pack_f16(x[6], x[7]));
            };
            for (int ch = tid; ch < 1024; ch += PREP_THREADS) {
                if (ch < 512) ainv_part(ch >> 3, (ch & 7) * 8);                          // P: rows 0..63, cols 0..63
                else ainv_part(64 + ((ch - 512) >> 3), 64 + ((ch - 512) & 7) * 8);       // Q: rows 64..127, cols 64..127
            }
            wait_mma();
            if (lq < 2) {
                float x[16];
                tmem_ld16(tmem + lane_off + 64u + (uint32_t)(cg * 16), x);
                tmem_ld_wait();
                if (FAST) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) x[j] *= sBeta[cg * 16 + j];
                }
#pragma unroll
                for (int j = 0; j < 16; j += 8)
                    sts_v4(sm, oY + sw128_off(64 + trow, cg * 16 + j, 128), pack_f16(x[j], x[j + 1]),
                           pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
            }
            if (tid < 512) {                 // zeros: rows 0..63, cols 64..127
                const int r = tid >> 3, c0 = 64 + (tid & 7) * 8;
                sts_v4(sm, oY + sw128_off(r, c0, 128), 0u, 0u, 0u, 0u);
            }
            sync_for_mma();

            // --------------------------------------------------------------
            // Phase 4: WY product (M=128, N=256, K=128) into TMEM [256,512):
            //   fast: Ainv diag(beta) [Lk | v]     (w still lacks diag(exp(P)))
            //   wide: Ainv [beta exp(G) k | beta v]
            // --------------------------------------------------------------
            if (tid == 0) {
                const Operand Ai{sbase + oY, false, 128}, Rh{sbase + (FAST ? 0u : wide_map::B2), true, 128};
                mma_128(tmem + 256, Ai, Rh, idesc_f16(T_F16, 128, 256, false, true), 8);
                mma_commit(bar);
            }
            // Meanwhile: A2 (inclusive lower) from TMEM [128,256) to fp16
            // K-major [t][i] in region W (the fp32 blocks are no longer needed).
            {
                float x[32];
                const int col0 = cg * 32;
                tmem_ld32(tmem + lane_off + 128u + (uint32_t)col0, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = (col0 + j <= trow) ? x[j] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    sts_v4(sm, RW + sw128_off(trow, col0 + j, 128), pack_f16(x[j], x[j + 1]), pack_f16(x[j + 2], x[j + 3]),
                           pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
            }
            wait_mma();
            // Phase 5: w | u from TMEM [256,512) to fp16 MN-major [t][n]
            // (fast: w columns scaled by exp(P)).
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                const int col0 = cg * 64 + part * 32;
                tmem_ld32(tmem + lane_off + 256u + (uint32_t)col0, x);
                tmem_ld_wait();
                if (FAST && col0 < 128) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] *= sEP[col0 + j];
                }
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    sts_v4(sm, (FAST ? 0u : wide_map::WU) + sw128_off(trow, col0 + j, 128), pack_f16(x[j], x[j + 1]),
                           pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
            }
            sync_for_mma();

            // --------------------------------------------------------------
            // Phase 6: [A2 w | A2 u] -> [256,512), then [X^T w | X^T u] ->
            // [0,256) with X = R (fast) or kg (wide).  Separate commits: the
            // epilogue of the first runs while the second computes.
            // --------------------------------------------------------------
            if (tid == 0) {
                const Operand KgT{sbase + (FAST ? oRf : wide_map::KGT), true, 128}, A2h{sbase + RW, false, 128},
                    WU{sbase + (FAST ? 0u : wide_map::WU), true, 128};
                mma_128(tmem + 256, A2h, WU, idesc_f16(T_F16, 128, 256, false, true), 8);
                mma_commit(bar);
                mma_128(tmem + 0, KgT, WU, idesc_f16(T_F16, 128, 256, true, true), 8);
                mma_commit(bar2);
            }
            wait_mma();

            // --------------------------------------------------------------
            // Phase 7 (fast kernel): epilogue through two 32 KB staging
            // buffers, one product at a time, each bulk-stored as soon as it
            // is staged; the buffer is reused once its store has read it.
            //   Qe = Lq diag(exp(P)) - A2 w -> ST1 (the A2 operand's region)
            //   [second product done: the next chunk's raw tiles are loaded
            //    into this chunk's w | u and inverse / R regions]
            //   Oi = A2 u -> ST0;  Nm = -cL R^T w -> ST1;  Bc = cL R^T u -> ST0
            // Thread w%4 lane quarter = row (t or d), columns 32 (w / 4) ..
            // --------------------------------------------------------------
            if constexpr (FAST) {
                uint8_t* dst = tile_ptr(p, c.slot, h);
                const ChunkRef& cx = have_n ? cn : none;
                const int col0 = cg * 32;
                float x[32];
                // Qe (rows t): qg from Lq (fp16) times exp(P), minus A2 w
                tmem_ld32(tmem + lane_off + 256u + (uint32_t)col0, x);
                tmem_ld_wait();
                load_g(cx, hn, 0);
                load_g(cx, hn, 1);
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    const uint4 qv = *reinterpret_cast<const uint4*>(sm + oRawQ + sw128_off(trow, col0 + j, 128));
                    float2 g0 = unpack_f16(qv.x), g1 = unpack_f16(qv.y), g2 = unpack_f16(qv.z), g3 = unpack_f16(qv.w);
                    const float4 e0 = *reinterpret_cast<const float4*>(sEP + col0 + j);
                    const float4 e1 = *reinterpret_cast<const float4*>(sEP + col0 + j + 4);
                    g0.x *= e0.x; g0.y *= e0.y; g1.x *= e0.z; g1.y *= e0.w;
                    g2.x *= e1.x; g2.y *= e1.y; g3.x *= e1.z; g3.y *= e1.w;
                    sts_v4(sm, ST1 + sw128_off(trow, col0 + j, 128), pack_f16(g0.x - x[j], g0.y - x[j + 1]),
                           pack_f16(g1.x - x[j + 2], g1.y - x[j + 3]), pack_f16(g2.x - x[j + 4], g2.y - x[j + 5]),
                           pack_f16(g3.x - x[j + 6], g3.y - x[j + 7]));
                }
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    bulk_s2g(dst + TILE_QE, sbase + ST1, BT * KD * 2);
                    bulk_commit();
                }
                load_g(cx, hn, 2);
                load_g(cx, hn, 3);
                // R^T [w | u] done: w | u, R and the inverse are free
                bounded_wait(bar2, phase2);
                phase2 ^= 1;
                tc_fence_after();
                if (tid == 0 && have_n) issue_raw(cn, hn, lay ^ 1);
                if (have_n) raw_pending = true;
                // Oi (rows t) -> its 32-column piece cg
                tmem_ld32(tmem + lane_off + 384u + (uint32_t)col0, x);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    sts_v4(sm, ST0 + (uint32_t)cg * OI_PIECE + sw64_off(trow, j), pack_f16(x[j], x[j + 1]),
                           pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]), pack_f16(x[j + 6], x[j + 7]));
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    bulk_s2g(dst + TILE_OI, sbase + ST0, NVT * OI_PIECE);
                    bulk_commit();
                    bulk_wait_read1();   // the Qe store has read ST1
                }
                load_beta(cx, hn);
                // Nm (rows d) = -cL R^T w
                const float rs = sCL[trow];
                tmem_ld32(tmem + lane_off + (uint32_t)col0, x);
                tmem_ld_wait();
                __syncthreads();
                {
                    const float ns = -rs;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, ST1 + sw128_off(trow, col0 + j, 128), pack_f16(ns * x[j], ns * x[j + 1]),
                               pack_f16(ns * x[j + 2], ns * x[j + 3]), pack_f16(ns * x[j + 4], ns * x[j + 5]),
                               pack_f16(ns * x[j + 6], ns * x[j + 7]));
                }
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    bulk_s2g(dst + TILE_NM, sbase + ST1, KD * KD * 2);
                    bulk_commit();
                    bulk_wait_read1();   // the Oi store has read ST0
                }
                // Bc (rows d) = cL R^T u -> its 32-column piece cg
                tmem_ld32(tmem + lane_off + 128u + (uint32_t)col0, x);
                tmem_ld_wait();
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 32; j += 8)
                    sts_v4(sm, ST0 + (uint32_t)cg * BC_PIECE + sw64_off(trow, j), pack_f16(rs * x[j], rs * x[j + 1]),
                           pack_f16(rs * x[j + 2], rs * x[j + 3]), pack_f16(rs * x[j + 4], rs * x[j + 5]),
                           pack_f16(rs * x[j + 6], rs * x[j + 7]));
                if (tid < 32) {
                    float4 dg;
                    dg.x = ex2(sGL[tid * 4 + 0]);
                    dg.y = ex2(sGL[tid * 4 + 1]);
                    dg.z = ex2(sGL[tid * 4 + 2]);
                    dg.w = ex2(sGL[tid * 4 + 3]);
                    *reinterpret_cast<float4*>(dst + TILE_DG + tid * 16) = dg;
                }
                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                if (tid == 0) {   // asynchronous: drains while the next chunk starts
                    bulk_s2g(dst + TILE_BC, sbase + ST0, NVT * BC_PIECE);
                    bulk_commit();
                }
            } else {
                // ----------------------------------------------------------
                // Phase 7 (wide kernel): epilogue in two stages.
                //   1. (first product done, the second still running)
                //      Qe = qg - A2 w -> ST_QE (Ainv's region),
                //      Oi = A2 u      -> ST_OI (A2's region); bulk-stored.
                //   2. (second product done)
                //      Nm = -kg^T w -> ST_NM, Bc = kg^T u -> ST_BC (over
                //      w | u); bulk-stored.  The next chunk's raw tiles
                //      (k over qg, v over kg, q over ST_QE) are requested
                //      once the Qe store has read its staging.
                // Lanes are rows (t for Qe / Oi, d for Nm / Bc); the four warps
                // of a lane quarter take one 32-column block of each product
                // (TMEM columns: Nm 0, Bc 128, Qe 256, Oi 384, + 32 role).
                // ----------------------------------------------------------
                uint8_t* dst = tile_ptr(p, c.slot, h);
                const int role = warp >> 2;
                const int col0 = role * 32;
                {
                    float x[32];
                    tmem_ld32(tmem + lane_off + 256u + (uint32_t)col0, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        const uint4 qv =
                            *reinterpret_cast<const uint4*>(sm + wide_map::QS + sw128_off(trow, col0 + j, 128));
                        const float2 g0 = unpack_f16(qv.x), g1 = unpack_f16(qv.y), g2 = unpack_f16(qv.z),
                                     g3 = unpack_f16(qv.w);
                        sts_v4(sm, wide_map::ST_QE + sw128_off(trow, col0 + j, 128),
                               pack_f16(g0.x - x[j], g0.y - x[j + 1]), pack_f16(g1.x - x[j + 2], g1.y - x[j + 3]),
                               pack_f16(g2.x - x[j + 4], g2.y - x[j + 5]), pack_f16(g3.x - x[j + 6], g3.y - x[j + 7]));
                    }
                    tmem_ld32(tmem + lane_off + 384u + (uint32_t)col0, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, wide_map::ST_OI + role * OI_PIECE + sw64_off(trow, j), pack_f16(x[j], x[j + 1]),
                               pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]),
                               pack_f16(x[j + 6], x[j + 7]));
                }
                fence_async_smem();
                __syncthreads();
                if (bulk_thread) {
                    bulk_s2g(dst + TILE_QE, sbase + wide_map::ST_QE, BT * KD * 2);
                    bulk_s2g(dst + TILE_OI, sbase + wide_map::ST_OI, NVT * OI_PIECE);
                    bulk_commit();
                }
                // the second product has read w | u and kg
                bounded_wait(bar2, phase2);
                phase2 ^= 1;
                tc_fence_after();
                {
                    float x[32];
                    // kg already carries exp(G_last - G): no row scale
                    tmem_ld32(tmem + lane_off + (uint32_t)col0, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, wide_map::ST_NM + sw128_off(trow, col0 + j, 128), pack_f16(-x[j], -x[j + 1]),
                               pack_f16(-x[j + 2], -x[j + 3]), pack_f16(-x[j + 4], -x[j + 5]),
                               pack_f16(-x[j + 6], -x[j + 7]));
                    tmem_ld32(tmem + lane_off + 128u + (uint32_t)col0, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        sts_v4(sm, wide_map::ST_BC + role * BC_PIECE + sw64_off(trow, j), pack_f16(x[j], x[j + 1]),
                               pack_f16(x[j + 2], x[j + 3]), pack_f16(x[j + 4], x[j + 5]),
                               pack_f16(x[j + 6], x[j + 7]));
                }
                if (tid < 32) {
                    float4 dg;
                    dg.x = ex2(sGL[tid * 4 + 0]);
                    dg.y = ex2(sGL[tid * 4 + 1]);
                    dg.z = ex2(sGL[tid * 4 + 2]);
                    dg.w = ex2(sGL[tid * 4 + 3]);
                    *reinterpret_cast<float4*>(dst + TILE_DG + tid * 16) = dg;
                }
                // the next chunk's gate rows and beta, as the fast epilogue loads them
                load_rows(have_n ? cn : none, hn);
                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                tc_fence_after();
                if (bulk_thread) {
                    bulk_s2g(dst + TILE_NM, sbase + wide_map::ST_NM, KD * KD * 2);
                    bulk_s2g(dst + TILE_BC, sbase + wide_map::ST_BC, NVT * BC_PIECE);
                    bulk_commit();
                    if (have_n) {
                        bulk_wait_read1();   // the Qe / Oi stores have read their staging
                        issue_raw(cn, hn, 0);
                    }
                }
                if (have_n) raw_pending = true;
            }
        }
        idx = nidx;
        item = nitem;
        c = cn;
        h = hn;
        have = have_n;
        if (FAST) lay ^= 1;   // the wide kernel keeps layout 0 (raw q at 64K)
    }
    if (bulk_thread) bulk_wait0();
    if (tid == 0) {
        if (*sFlag != 0) atomicOr(p.status, STATUS_TIMEOUT);
        // a chunk's raw tiles issued before the loop ended (after a timeout)
        // have landed before the shared memory is released
        if (raw_pending) mbar_wait(rawbar, rphase, DRAIN_LIMIT);
        // every product this thread issued has completed before TMEM is freed
        mma_commit(sbase + M_BARD);
        mbar_wait(sbase + M_BARD, 0, DRAIN_LIMIT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

namespace {

// The driver's tensor-map encoder, found once through the runtime (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// q, k or v ([tokens][H][128] bf16) as a 3-D tensor (dimension, head, token):
// one load brings 64 dimensions of one head for 128 consecutive tokens, in
// the 128-byte swizzled layout of the MMA operands; tokens past the end read
// as zero.
bool make_row_map(CUtensorMap* m, const void* base, int H, long long ntok) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)ntok};
    const cuuint64_t strides[2] = {(cuuint64_t)KD * 2u, (cuuint64_t)H * KD * 2u};
    const cuuint32_t box[3] = {64u, 1u, (cuuint32_t)BT};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <bool L2NORM, bool FAST>
static cudaError_t launch_one(const FwdParams& p, const CUtensorMap (&tm)[3], unsigned grid, cudaStream_t stream) {
    cudaError_t e =
        cudaFuncSetAttribute(kda_prep_kernel<L2NORM, FAST>, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
    if (e != cudaSuccess) return e;
    kda_prep_kernel<L2NORM, FAST><<<grid, PREP_THREADS, PREP_SMEM, stream>>>(p, tm[0], tm[1], tm[2]);
    return cudaGetLastError();
}

// Host-side launcher: the fast kernel over every work item, then the wide
// kernel over whatever the fast one queued (usually nothing; its CTAs then
// exit at once).  One persistent CTA per SM, fewer if there is less work.
cudaError_t launch_prep(const FwdParams& p, bool l2norm, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long items = (long long)p.nslots * p.H;
    const unsigned grid = (unsigned)(items < sms ? items : sms);
    if (grid == 0) return cudaSuccess;
    const long long ntok = p.cu != nullptr ? (long long)p.T : (long long)p.N * p.T;
    if (ntok == 0) return cudaSuccess;   // no tokens: every chunk slot is empty
    CUtensorMap tm[3];
    if (!make_row_map(&tm[0], p.q, p.H, ntok) || !make_row_map(&tm[1], p.k, p.H, ntok) ||
        !make_row_map(&tm[2], p.v, p.H, ntok))
        return cudaErrorInvalidValue;
    e = l2norm ? launch_one<true, true>(p, tm, grid, stream) : launch_one<false, true>(p, tm, grid, stream);
    if (e != cudaSuccess) return e;
    return l2norm ? launch_one<true, false>(p, tm, grid, stream) : launch_one<false, false>(p, tm, grid, stream);
}

}  // namespace kda
