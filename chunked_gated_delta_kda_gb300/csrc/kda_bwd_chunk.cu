// Chunk-parallel KDA backward.
//
// The forward in the transition form (section "算法原理" M4 of the page
// "PyPTO-Gym chunk_kda operator: an NPU forward of chunked gated delta-rule
// linear attention"), per 128-token chunk c with entering state S_c (K x V):
//   S_{c+1} = Dg_c * S_c + Nm_c S_c + Bc_c,     o_c = Qe_c S_c + Oi_c
// so the state gradient obeys, from dS_N = dht backwards,
//   dS_c = Dg_c * dS_{c+1} + Nm_c^T dS_{c+1} + Qe_c^T do_c.
// That is the forward's state recurrence again, on the tiles (Nm^T, Qe^T do,
// Dg) in reverse chunk order.  kda_bwd_tiles_kernel builds those tiles from
// the forward's; the forward's scan kernel then runs it (state-only mode) and
// stores dS_{c+1} for every chunk.  With S_c (stored by the forward scan) and
// dS_{c+1} known, every chunk is independent: kda_bwd_chunk_kernel replays
// its 128 tokens forward in fp32 and applies the per-token chain rule
// backwards (the same rule as the token-by-token backward kernel).
//
// Replaying backwards needs the state entering each token.  The kernel keeps
// the delta residual r_t = v_t - k_t.(exp(g_t) S_{t-1}) of every token (64
// KiB of shared memory per chunk) and a copy of the state every 16 tokens
// (in a per-CTA global scratch that stays in L2), and reconstructs
//   exp(g_t) S_{t-1} = S_t - beta_t k_t r_t^T,   S_{t-1} = exp(-g_t) (that)
// which multiplies rounding errors by exp(-g) per token; the 16-token copies
// bound the growth to exp(sum of -g over 16 tokens).  A chunk where that sum
// exceeds EXACT_WINDOW_DECAY in some dimension stores the state entering
// every token instead (8 MiB of scratch) and needs no division.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda.h"
#include "kda_bwd.cuh"
#include "kda_common.cuh"
#include "sm100_ptx.cuh"
#include "kda_mma_tf32.cuh"

namespace kda {

namespace {

// ---------------------------------------------------------------------------
// Transposed tiles
// ---------------------------------------------------------------------------
constexpr int BT_THREADS = 256;
// Shared memory (1024-aligned): the forward's Qe tile as stored (fp16, 128-byte
// swizzled [t][d]: the MN-major A operand of Qe^T), the raw Nm tile, do as fp16
// in the same layout (the MN-major B operand), then barriers and scratch.
constexpr uint32_t BTS_QE = 0, BTS_NM = 32768, BTS_DO = 65536, BTS_MISC = 98304;
constexpr uint32_t BTS_BAR_TX = BTS_MISC, BTS_BAR_MMA = BTS_MISC + 8, BTS_TMEM = BTS_MISC + 16,
                   BTS_MAX = BTS_MISC + 32;   // f32[8]: per-warp max |do|
constexpr uint32_t BT_SMEM = BTS_MISC + 64 + 1024;

__device__ __forceinline__ uint32_t f2h(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace

// One CTA per (chunk slot, head), two CTAs per SM: writes, at the mirrored
// chunk position of the same sequence, the tile the reverse state pass reads:
// Nm^T (same fp16 128-byte-swizzled layout as Nm), Qe^T do as the four fp16
// Bc pieces, Dg.  Qe^T do is one M=128 N=128 K=128 tcgen05 product (fp16
// operands, fp32 accumulation in TMEM).  do enters as fp16 scaled by a power
// of two, 2^s with s from the chunk's largest |do|, so that the bf16 -> fp16
// conversion is exact in range; the accumulator is multiplied by 2^-s.
__global__ void __launch_bounds__(BT_THREADS, 2) kda_bwd_tiles_kernel(const FwdParams fp, uint8_t* btiles,
                                                                      const uint16_t* __restrict__ dout) {
    extern __shared__ uint8_t bsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(bsm_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int slot = (int)blockIdx.x, h = (int)blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = fp.H;
    ChunkRef c;
    if (!slot_chunk(fp, slot, c)) return;   // uniform
    long long bos;
    int len;
    if (!seq_bounds(fp, c.n, bos, len)) return;
    const int nch = (len + BT - 1) / BT;
    const uint8_t* src = tile_ptr(fp, slot, h);
    uint8_t* dst = btiles + ((size_t)chunk_slot(fp, c.n, nch - 1 - c.j) * H + h) * TILE_BYTES;
    const uint32_t bar_tx = sbase + BTS_BAR_TX, bar_mma = sbase + BTS_BAR_MMA;
    float* wmax = reinterpret_cast<float*>(sm + BTS_MAX);

    if (tid == 0) {
        mbar_init(bar_tx, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(sbase + BTS_TMEM, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + BTS_TMEM);
    if (tid == 0) {   // the forward's Nm and Qe tiles, as stored
        mbar_arrive_expect_tx(bar_tx, 65536u);
        bulk_g2s(sbase + BTS_NM, src + TILE_NM, 32768u, bar_tx);
        bulk_g2s(sbase + BTS_QE, src + TILE_QE, 32768u, bar_tx);
    }
    if (tid < KD / 4)
        reinterpret_cast<float4*>(dst + TILE_DG)[tid] = reinterpret_cast<const float4*>(src + TILE_DG)[tid];

    // do of the chunk's rows: 8 pieces of 8 values per thread (rows past the
    // chunk's length are zero), and the chunk's largest |do|
    uint4 dr[8];
    float m = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = tid + u * BT_THREADS, t = i >> 4, c8 = (i & 15) * 8;
        dr[u] = make_uint4(0u, 0u, 0u, 0u);
        if (t < c.len) dr[u] = *reinterpret_cast<const uint4*>(dout + ((size_t)(c.tok0 + t) * H + h) * VD + c8);
        const uint32_t w4[4] = {dr[u].x, dr[u].y, dr[u].z, dr[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)   // |x| of the two bf16 halves as fp32 bit patterns
            m = fmaxf(m, fmaxf(__uint_as_float((w4[e] << 16) & 0x7fff0000u), __uint_as_float(w4[e] & 0x7fff0000u)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) wmax[warp] = m;
    __syncthreads();
    m = wmax[0];
#pragma unroll
    for (int w = 1; w < BT_THREADS / 32; ++w) m = fmaxf(m, wmax[w]);
    // 2^s brings the largest |do| into [2^13, 2^14); |s| <= 126 keeps 2^s and 2^-s normal
    int s = 0;
    if (m > 0.f && m <= 3.0e38f) s = 13 - (int)((__float_as_uint(m) >> 23) & 0xffu) + 127;
    s = s < -126 ? -126 : (s > 126 ? 126 : s);
    const float up = __uint_as_float((uint32_t)(s + 127) << 23), down = __uint_as_float((uint32_t)(127 - s) << 23);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = tid + u * BT_THREADS, t = i >> 4, c8 = (i & 15) * 8;
        const uint32_t w4[4] = {dr[u].x, dr[u].y, dr[u].z, dr[u].w};
        uint32_t o4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o4[e] = f2h(__uint_as_float(w4[e] << 16) * up, __uint_as_float(w4[e] & 0xffff0000u) * up);
        *reinterpret_cast<uint4*>(sm + BTS_DO + sw128_off(t, c8, 128)) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
    fence_async_smem();
    const bool tx_done = __syncthreads_and(mbar_wait(bar_tx, 0, wait_limit_of(fp))) != 0;
    tc_fence_after();
    bool ok = tx_done;
    if (ok && warp == 0) {   // Bq[d][v] = sum_t Qe[t][d] do[t][v]: both operands MN-major, K = t
        const uint64_t da = smem_desc(sbase + BTS_QE, 16384u, 1024u, SW_128B);
        const uint64_t db = smem_desc(sbase + BTS_DO, 16384u, 1024u, SW_128B);
        const uint32_t id = idesc_f16(T_F16, 128, 128, true, true);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_f16_warp(tmem, da + (uint64_t)ks * 128u, db + (uint64_t)ks * 128u, id, ks > 0);
        mma_commit_warp(bar_mma);
    }

    // Nm^T while the product runs: write (d, e) <- Nm(e, d) in 16-byte runs.
    // The lanes sharing d read rows e0 + u with e0 a multiple of 8, which
    // all fall on one swizzled 16-byte position; each lane therefore starts
    // at its own u (k = e0 / 8 % 8: 2-way instead of 16-way bank conflicts)
    // and rotates its eight values back into place.
    if (ok) {
        const uint8_t* raw = sm + BTS_NM;
        for (int i = tid; i < KD * KD / 8; i += BT_THREADS) {
            const int d = i >> 4, e0 = (i & 15) * 8, k = i & 7;
            uint32_t x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)   // x[u] = Nm(e0 + (u + k) % 8, d)
                x[u] = *reinterpret_cast<const uint16_t*>(raw + sw128_off(e0 + ((u + k) & 7), d, 128));
#pragma unroll
            for (int b = 1; b < 8; b <<= 1) {   // rotate by k: x[j] <- x[(j - k) % 8]
                if (k & b) {
                    uint32_t y[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) y[j] = x[(j - b) & 7];
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = y[j];
                }
            }
            *reinterpret_cast<uint4*>(dst + TILE_NM + sw128_off(d, e0, 128)) =
                make_uint4(x[0] | (x[1] << 16), x[2] | (x[3] << 16), x[4] | (x[5] << 16), x[6] | (x[7] << 16));
        }
    }

    // Bq rows d = TMEM lanes; warp w reads lane quarter w % 4, columns 64 (w / 4) ..
    // +64, i.e. two of the four 32-column Bc pieces
    bool mma_done = false;
    if (ok) ok = mma_done = __syncthreads_and(mbar_wait(bar_mma, 0, wait_limit_of(fp))) != 0;
    tc_fence_after();
    if (ok) {
        const int d = 32 * (warp & 3) + lane;
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
            const int vt = 2 * (warp >> 2) + q;
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(vt * BV), x);
            tmem_ld_wait();
            uint8_t* piece = dst + TILE_BC + vt * BC_PIECE;
#pragma unroll
            for (int j = 0; j < BV; j += 8)
                *reinterpret_cast<uint4*>(piece + sw64_off(d, j)) =
                    make_uint4(f2h(x[j] * down, x[j + 1] * down), f2h(x[j + 2] * down, x[j + 3] * down),
                               f2h(x[j + 4] * down, x[j + 5] * down), f2h(x[j + 6] * down, x[j + 7] * down));
        }
    } else {   // a bounded wait ran out: flag it, let the copies and the product finish (bounded), free TMEM
        if (tid == 0) atomicOr(fp.status, STATUS_TIMEOUT);
        if (!tx_done) mbar_wait(bar_tx, 0, DRAIN_LIMIT);
        else if (!mma_done) mbar_wait(bar_mma, 0, DRAIN_LIMIT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// Chunk-local backward
// ---------------------------------------------------------------------------
namespace {

constexpr int CB_THREADS = 512;
constexpr int CB_WARPS = CB_THREADS / 32;
constexpr int CB_ROWS = 8;
constexpr int CB_RED = 3 * KD + 4;
constexpr int CB_WIN = 16;                          // tokens between stored states
constexpr float EXACT_WINDOW_DECAY = 7.0f;          // max sum of -g over a window before exact mode
constexpr uint32_t CB_RED_BYTES = 2u * CB_WARPS * CB_RED * 4u;
// Per-warp ring of token inputs, filled by cp.async CB_AHEAD tokens ahead of
// use: q (256 B) | k (256 B) | g (512 B) | the warp's 8 v (16 B) | 8 do (16 B) | beta.
constexpr int CB_RING = 4;
constexpr int CB_AHEAD = 2;
constexpr uint32_t TS_Q = 0, TS_K = 256, TS_G = 512, TS_V = 1024, TS_DO = 1040, TS_B = 1056, TS_BYTES = 1072;
constexpr uint32_t CB_RING_BYTES = (uint32_t)CB_WARPS * CB_RING * TS_BYTES;
constexpr uint32_t CB_SMEM = CB_RED_BYTES + BT * VD * 4u + CB_RING_BYTES;   // + residuals r[t][v] + rings

struct Tok {
    float q[4], k[4], e[4], ie[4];
    float beta;
    float v[CB_ROWS];
};

__device__ __forceinline__ void rows8_bf16(const uint16_t* p, float (&x)[CB_ROWS]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
    x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
    x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_ahead() {
    asm volatile("cp.async.wait_group %0;" ::"n"(CB_AHEAD) : "memory");
}

// Copy one token's inputs into a ring slot (every lane issues its share).
__device__ __forceinline__ void tok_fetch(const BwdParams& p, size_t tok, int v0, int lane, uint32_t slot) {
    if (lane < 16) cp_async16(slot + TS_Q + 16u * lane, p.q + tok * KD + 8 * lane);
    else cp_async16(slot + TS_K + 16u * (lane - 16), p.k + tok * KD + 8 * (lane - 16));
    cp_async16(slot + TS_G + 16u * lane, p.g + tok * KD + 4 * lane);
    if (lane == 0) cp_async16(slot + TS_V, p.v + tok * VD + v0);
    if (lane == 1) cp_async16(slot + TS_DO, p.dout + tok * VD + v0);
    if (lane == 2) cp_async4(slot + TS_B, p.beta + tok);
}

// A token's inputs from its ring slot (generic pointer `ts`).
__device__ __forceinline__ void tok_load(const BwdParams& p, const uint8_t* ts, int lane, Tok& in) {
    load4_bf16(reinterpret_cast<const uint16_t*>(ts + TS_Q) + 4 * lane, in.q);
    load4_bf16(reinterpret_cast<const uint16_t*>(ts + TS_K) + 4 * lane, in.k);
    const float4 gv = *reinterpret_cast<const float4*>(ts + TS_G + 16 * lane);
    in.beta = *reinterpret_cast<const float*>(ts + TS_B);
    rows8_bf16(reinterpret_cast<const uint16_t*>(ts + TS_V), in.v);
    float qs = p.scale, ks = 1.f;
    if (p.l2norm) {   // x / sqrt(sum x^2 + 1e-6), section "测试与验证体系"
        const float sq = warp_sum(in.q[0] * in.q[0] + in.q[1] * in.q[1] + in.q[2] * in.q[2] + in.q[3] * in.q[3]);
        const float sk = warp_sum(in.k[0] * in.k[0] + in.k[1] * in.k[1] + in.k[2] * in.k[2] + in.k[3] * in.k[3]);
        qs *= rsqrtf(sq + 1e-6f);
        ks = rsqrtf(sk + 1e-6f);
    }
    const float g[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        in.q[i] *= qs;
        in.k[i] *= ks;
        in.e[i] = __expf(g[i]);
        in.ie[i] = __expf(-g[i]);
    }
}

// state rows v0..v0+7, K entries 4 lane..+3, from a [K][V] fp32 slab
__device__ __forceinline__ void load_kv(const float* slab, int v0, int lane, float (&s)[CB_ROWS][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 a = *reinterpret_cast<const float4*>(slab + (size_t)(4 * lane + i) * VD + v0);
        const float4 b = *reinterpret_cast<const float4*>(slab + (size_t)(4 * lane + i) * VD + v0 + 4);
        s[0][i] = a.x; s[1][i] = a.y; s[2][i] = a.z; s[3][i] = a.w;
        s[4][i] = b.x; s[5][i] = b.y; s[6][i] = b.z; s[7][i] = b.w;
    }
}

// own entries of a [V][K] fp32 state (each thread reads back what it wrote)
__device__ __forceinline__ void put_vk(float* slab, int v0, int lane, const float (&s)[CB_ROWS][4]) {
#pragma unroll
    for (int r = 0; r < CB_ROWS; ++r)
        *reinterpret_cast<float4*>(slab + (size_t)(v0 + r) * KD + 4 * lane) = make_float4(s[r][0], s[r][1], s[r][2], s[r][3]);
}
__device__ __forceinline__ void get_vk(const float* slab, int v0, int lane, float (&s)[CB_ROWS][4]) {
#pragma unroll
    for (int r = 0; r < CB_ROWS; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(slab + (size_t)(v0 + r) * KD + 4 * lane);
        s[r][0] = x.x; s[r][1] = x.y; s[r][2] = x.z; s[r][3] = x.w;
    }
}

}  // namespace

__global__ void __launch_bounds__(CB_THREADS, 1) kda_bwd_chunk_kernel(const BwdParams p, const FwdParams fp) {
    extern __shared__ __align__(16) float csm[];
    float* red = csm;                                   // [2][CB_WARPS][CB_RED]
    float* rres = csm + CB_RED_BYTES / 4;               // [BT][VD]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = reinterpret_cast<uint8_t*>(csm) + CB_RED_BYTES + BT * VD * 4u + (size_t)warp * CB_RING * TS_BYTES;
    const uint32_t ring_s = smem_u32(ring);
    const int v0 = warp * CB_ROWS;
    const int H = p.H;
    const long long items = (long long)fp.nslots * H;
    float* scratch = p.scratch + (size_t)blockIdx.x * BT * VD * KD;

    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        if (p.tc_skip != nullptr && p.tc_skip[it] == 0u) continue;   // done by the tensor-core kernel
        const int slot = (int)(it / H), h = (int)(it % H);
        ChunkRef c;
        if (!slot_chunk(fp, slot, c)) continue;                    // uniform
        if (fp.exact_flags[(size_t)c.n * H + h] != 0u) continue;   // replayed by the token-by-token kernel
        long long bos;
        int len;
        if (!seq_bounds(fp, c.n, bos, len)) continue;
        const int nch = (len + BT - 1) / BT;
        const int rows = c.len;

        // window decay check: warp w < 8 sums max(-g, 0) over tokens [16 w, 16 w + 16)
        bool big = false;
        if (warp < BT / CB_WIN) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int t = warp * CB_WIN; t < min(rows, (warp + 1) * CB_WIN); ++t) {
                const float4 gv = *reinterpret_cast<const float4*>(p.g + ((size_t)(c.tok0 + t) * H + h) * KD + 4 * lane);
                acc[0] += fmaxf(-gv.x, 0.f); acc[1] += fmaxf(-gv.y, 0.f);
                acc[2] += fmaxf(-gv.z, 0.f); acc[3] += fmaxf(-gv.w, 0.f);
            }
            big = fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])) > EXACT_WINDOW_DECAY ||
                  !(acc[0] + acc[1] + acc[2] + acc[3] < 3.0e38f);
        }
        const int win = __syncthreads_or(big) ? 1 : CB_WIN;

        // Token inputs stream through the warp's ring in the order the two
        // phases use them: t = 0 .. rows-1, then rows-1 .. 0 (step i).
        const int steps = 2 * rows;
        auto fetch = [&](int i) {
            if (i < steps) {
                const int t = i < rows ? i : steps - 1 - i;
                tok_fetch(p, (size_t)(c.tok0 + t) * H + h, v0, lane, ring_s + (uint32_t)(i % CB_RING) * TS_BYTES);
            }
            cp_async_commit();   // one group per step, empty past the end
        };
        auto slot_of = [&](int i) -> const uint8_t* {
            __syncwarp();
            fetch(i + CB_AHEAD);   // the slot it fills was last read at step i + CB_AHEAD - CB_RING < i
            cp_async_wait_ahead();
            __syncwarp();
            return ring + (size_t)(i % CB_RING) * TS_BYTES;
        };
        for (int i = 0; i < CB_AHEAD; ++i) fetch(i);

        // phase A: replay the chunk forward from S_c, keeping r_t and the stored states
        float s[CB_ROWS][4];
        load_kv(p.ckpt_s + ((size_t)slot * H + h) * KD * VD, v0, lane, s);
        for (int t = 0; t < rows; ++t) {
            if (t % win == 0) put_vk(scratch + (size_t)(t / win) * VD * KD, v0, lane, s);
            Tok in;
            tok_load(p, slot_of(t), lane, in);
            float dot[CB_ROWS];
#pragma unroll
            for (int r = 0; r < CB_ROWS; ++r) {
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
            for (int r = 0; r < CB_ROWS; ++r) {
                dot[r] = in.v[r] - dot[r];
                const float br = in.beta * dot[r];
#pragma unroll
                for (int i = 0; i < 4; ++i) s[r][i] = fmaf(in.k[i], br, s[r][i]);
            }
            if (lane == 0) {
                float4* rr = reinterpret_cast<float4*>(rres + (size_t)t * VD + v0);
                rr[0] = make_float4(dot[0], dot[1], dot[2], dot[3]);
                rr[1] = make_float4(dot[4], dot[5], dot[6], dot[7]);
            }
        }
        __syncthreads();

        // phase B: the chain rule backwards from dS_{c+1}
        float d[CB_ROWS][4];
        load_kv(p.ckpt_d + ((size_t)chunk_slot(fp, c.n, nch - 1 - c.j) * H + h) * KD * VD, v0, lane, d);
        for (int t = rows - 1; t >= 0; --t) {
            const size_t tok = (size_t)(c.tok0 + t) * H + h;
            Tok in;
            const uint8_t* ts = slot_of(steps - 1 - t);
            tok_load(p, ts, lane, in);
            float dov[CB_ROWS], rr[CB_ROWS], gk[CB_ROWS];
            rows8_bf16(reinterpret_cast<const uint16_t*>(ts + TS_DO), dov);
            {
                const float4 a = *reinterpret_cast<const float4*>(rres + (size_t)t * VD + v0);
                const float4 b = *reinterpret_cast<const float4*>(rres + (size_t)t * VD + v0 + 4);
                rr[0] = a.x; rr[1] = a.y; rr[2] = a.z; rr[3] = a.w; rr[4] = b.x; rr[5] = b.y; rr[6] = b.z; rr[7] = b.w;
            }
            float pdq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < CB_ROWS; ++r) {
                const float br = in.beta * rr[r];
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pdq[i] = fmaf(dov[r], s[r][i], pdq[i]);        // do_v s_v'
                    s[r][i] = fmaf(-br, in.k[i], s[r][i]);          // a_v = s_v' - beta r_v k
                    d[r][i] = fmaf(dov[r], in.q[i], d[r][i]);       // G_v
                    acc = fmaf(d[r][i], in.k[i], acc);
                }
                gk[r] = acc;
            }
            warp_sum8(gk, lane);
            float pdk[4] = {0.f, 0.f, 0.f, 0.f}, pdg[4] = {0.f, 0.f, 0.f, 0.f};
            float pdb = 0.f;
#pragma unroll
            for (int r = 0; r < CB_ROWS; ++r) {
                pdb = fmaf(rr[r], gk[r], pdb);
                const float bg = in.beta * gk[r];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pdk[i] = fmaf(rr[r], d[r][i], fmaf(-gk[r], s[r][i], pdk[i]));
                    d[r][i] = fmaf(-bg, in.k[i], d[r][i]);          // dA_v
                    pdg[i] = fmaf(d[r][i], s[r][i], pdg[i]);
                    d[r][i] *= in.e[i];                              // dL/ds_v before the token
                }
            }
            if (lane < 2) {
                const int r0 = 4 * lane;
                *reinterpret_cast<float4*>(p.dv + tok * VD + v0 + r0) =
                    make_float4(in.beta * gk[r0], in.beta * gk[r0 + 1], in.beta * gk[r0 + 2], in.beta * gk[r0 + 3]);
            }
            // the state entering token t: stored, or exp(-g) a
            if (t % win == 0) {
                if (t > 0) get_vk(scratch + (size_t)(t / win) * VD * KD, v0, lane, s);
            } else {
#pragma unroll
                for (int r = 0; r < CB_ROWS; ++r)
#pragma unroll
                    for (int i = 0; i < 4; ++i) s[r][i] *= in.ie[i];
            }
            float* buf = red + ((size_t)(t & 1) * CB_WARPS + warp) * CB_RED;
            *reinterpret_cast<float4*>(buf + 4 * lane) = make_float4(pdq[0], pdq[1], pdq[2], pdq[3]);
            *reinterpret_cast<float4*>(buf + KD + 4 * lane) = make_float4(pdk[0], pdk[1], pdk[2], pdk[3]);
            *reinterpret_cast<float4*>(buf + 2 * KD + 4 * lane) = make_float4(pdg[0], pdg[1], pdg[2], pdg[3]);
            if (lane == 0) buf[3 * KD] = pdb;
            __syncthreads();
            const int i = threadIdx.x;
            if (i <= 3 * KD) {
                const float* col = red + (size_t)(t & 1) * CB_WARPS * CB_RED + i;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < CB_WARPS; ++w) sum += col[(size_t)w * CB_RED];
                if (i < KD) p.dq[tok * KD + i] = p.scale * sum;
                else if (i < 2 * KD) p.dk[tok * KD + i - KD] = in.beta * sum;
                else if (i < 3 * KD) p.dg[tok * KD + i - 2 * KD] = sum;
                else p.dbeta[tok] = sum;
            }
        }
        __syncthreads();   // this chunk's last reduction and residuals are read
    }
}

cudaError_t launch_bwd_tiles(const FwdParams& fp, uint8_t* btiles, const uint16_t* dout, cudaStream_t stream) {
    if (fp.nslots == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BT_SMEM);
    if (e != cudaSuccess) return e;
    kda_bwd_tiles_kernel<<<dim3((unsigned)fp.nslots, (unsigned)fp.H), BT_THREADS, BT_SMEM, stream>>>(fp, btiles, dout);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunk(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream) {
    if (fp.nslots == 0 || ctas == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CB_SMEM);
    if (e != cudaSuccess) return e;
    kda_bwd_chunk_kernel<<<ctas, CB_THREADS, CB_SMEM, stream>>>(p, fp);
    return cudaGetLastError();
}

}  // namespace kda
