// Sequential half of the chunked KDA forward ("scan"): for one (sequence,
// head, 32-wide value tile) it walks the chunks in order carrying the state
// S (K x 32, fp32, one row per thread) and produces the output rows:
//   S' = Dg * S + Nm S + Bc,     o = Qe S + Oi
// which is step M4 of the page "PyPTO-Gym chunk_kda operator: an NPU forward
// of chunked gated delta-rule linear attention" (section "算法原理") in the
// exact re-associated form set out in kda_common.cuh.  The initial and final
// states use the page's [N, H, V, K] layout (section "算子签名与 I/O 规格"),
// i.e. the transpose of the K x V state; the transpose happens here.
//
// GB300 mapping.  128 threads; thread i owns state row d = i and output row
// t = i (TMEM lane i).  Per chunk, two M=128 N=32 K=128 fp16 MMAs (Nm S and
// Qe S) read the fp16 copy of S from shared memory and accumulate in TMEM;
// the fp32 state update, Bc / Oi additions and the bf16 output conversion
// run on CUDA cores.  The chunk tiles are double-buffered with 1-D bulk
// copies so that chunk j+1's tiles land while chunk j computes.
#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int SCAN_THREADS = 128;
constexpr uint32_t ST_NM = 0;
constexpr uint32_t ST_QE = 32768;
constexpr uint32_t ST_BC = 65536;
constexpr uint32_t ST_OI = 73728;
constexpr uint32_t ST_DG = 81920;
constexpr uint32_t ST_BYTES = 82432;          // bytes loaded per stage
constexpr uint32_t ST_STRIDE = 82944;         // 1024-aligned stage stride
constexpr uint32_t S_S16 = 2 * ST_STRIDE;     // fp16 state copy, [K][32] 64B-swizzled
constexpr uint32_t S_BAR = S_S16 + 8192;      // full[2], mma
constexpr uint32_t S_TMEM = S_BAR + 64;
constexpr uint32_t S_FLAG = S_TMEM + 4;
constexpr uint32_t SCAN_SMEM = S_BAR + 128 + 1024;

__device__ __forceinline__ void load_stage(const FwdParams& p, int slot, int h, int vt, uint32_t dst,
                                           uint32_t bar) {
    const uint8_t* src = tile_ptr(p, slot, h);
    mbar_arrive_expect_tx(bar, ST_BYTES);
    bulk_g2s(dst + ST_NM, src + TILE_NM, KD * KD * 2, bar);
    bulk_g2s(dst + ST_QE, src + TILE_QE, BT * KD * 2, bar);
    bulk_g2s(dst + ST_BC, src + TILE_BC + vt * BC_PIECE, BC_PIECE, bar);
    bulk_g2s(dst + ST_OI, src + TILE_OI + vt * OI_PIECE, OI_PIECE, bar);
    bulk_g2s(dst + ST_DG, src + TILE_DG, KD * 4, bar);
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
}

}  // namespace

__global__ void __launch_bounds__(SCAN_THREADS, 1) kda_scan_kernel(const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int vt = (int)blockIdx.x;
    const int h = (int)blockIdx.y;
    const int n = (int)blockIdx.z;
    const int H = p.H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;

    long long bos;
    int len;
    if (!seq_bounds(p, n, bos, len)) return;        // uniform
    const int nch = (len + BT - 1) / BT;

    const uint32_t full0 = sbase + S_BAR, full1 = sbase + S_BAR + 8, mbar = sbase + S_BAR + 16;
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(sm + S_FLAG);
    if (warp == 0) {
        tmem_alloc(sbase + S_TMEM, 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(full0, 1);
        mbar_init(full1, 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
        *sFlag = 0;
    }

    // State rows: thread d holds S[d][vt*32 .. vt*32+31] (fp32).
    const int d = tid;
    float S[BV];
    const size_t sbase_state = ((size_t)n * H + h) * VD * KD;   // [N,H,V,K] slab
    if (p.h0 != nullptr) {
#pragma unroll
        for (int j = 0; j < BV; ++j) S[j] = __ldg(p.h0 + sbase_state + (size_t)(vt * BV + j) * KD + d);
    } else {
#pragma unroll
        for (int j = 0; j < BV; ++j) S[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < BV; j += 8)
        *reinterpret_cast<uint4*>(sm + S_S16 + sw64_off(d, j)) =
            make_uint4(pack_f16x2(S[j], S[j + 1]), pack_f16x2(S[j + 2], S[j + 3]), pack_f16x2(S[j + 4], S[j + 5]),
                       pack_f16x2(S[j + 6], S[j + 7]));
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + S_TMEM);
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    if (tid == 0) {
        if (nch > 0) load_stage(p, chunk_slot(p, n, 0), h, vt, sbase + 0 * ST_STRIDE, full0);
        if (nch > 1) load_stage(p, chunk_slot(p, n, 1), h, vt, sbase + 1 * ST_STRIDE, full1);
    }

    const uint32_t id = idesc_f16(T_F16, 128, BV, false, true);
    for (int j = 0; j < nch; ++j) {
        const int s = j & 1;
        const uint32_t stage = sbase + (uint32_t)s * ST_STRIDE;
        const uint8_t* st = sm + (size_t)s * ST_STRIDE;
        if (!mbar_wait(s ? full1 : full0, (uint32_t)(j >> 1) & 1u, WAIT_LIMIT)) *sFlag = 1;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t bdesc = smem_desc(sbase + S_S16 + (uint32_t)ks * 1024u, 512u, 512u, SW_64B);
                const uint64_t a_nm = smem_desc(stage + ST_NM + (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u,
                                                16u, 1024u, SW_128B);
                const uint64_t a_qe = smem_desc(stage + ST_QE + (uint32_t)(ks >> 2) * 16384u + (uint32_t)(ks & 3) * 32u,
                                                16u, 1024u, SW_128B);
                mma_f16(tmem + 0, a_nm, bdesc, id, ks > 0);
                mma_f16(tmem + BV, a_qe, bdesc, id, ks > 0);
            }
            mma_commit(mbar);
        }
        if (!mbar_wait(mbar, (uint32_t)j & 1u, WAIT_LIMIT)) *sFlag = 1;
        tc_fence_after();

        // State update, row d = tid.
        {
            float x[BV];
            tmem_ld32(tmem + lane_off + 0u, x);
            tmem_ld_wait();
            const float Dd = *reinterpret_cast<const float*>(st + ST_DG + d * 4);
#pragma unroll
            for (int c8 = 0; c8 < BV; c8 += 8) {
                const uint4 b = *reinterpret_cast<const uint4*>(st + ST_BC + sw64_off(d, c8));
                const float2 b0 = unpack_f16x2(b.x), b1 = unpack_f16x2(b.y), b2 = unpack_f16x2(b.z),
                             b3 = unpack_f16x2(b.w);
                S[c8 + 0] = fmaf(Dd, S[c8 + 0], x[c8 + 0] + b0.x);
                S[c8 + 1] = fmaf(Dd, S[c8 + 1], x[c8 + 1] + b0.y);
                S[c8 + 2] = fmaf(Dd, S[c8 + 2], x[c8 + 2] + b1.x);
                S[c8 + 3] = fmaf(Dd, S[c8 + 3], x[c8 + 3] + b1.y);
                S[c8 + 4] = fmaf(Dd, S[c8 + 4], x[c8 + 4] + b2.x);
                S[c8 + 5] = fmaf(Dd, S[c8 + 5], x[c8 + 5] + b2.y);
                S[c8 + 6] = fmaf(Dd, S[c8 + 6], x[c8 + 6] + b3.x);
                S[c8 + 7] = fmaf(Dd, S[c8 + 7], x[c8 + 7] + b3.y);
            }
#pragma unroll
            for (int c8 = 0; c8 < BV; c8 += 8)
                *reinterpret_cast<uint4*>(sm + S_S16 + sw64_off(d, c8)) =
                    make_uint4(pack_f16x2(S[c8], S[c8 + 1]), pack_f16x2(S[c8 + 2], S[c8 + 3]),
                               pack_f16x2(S[c8 + 4], S[c8 + 5]), pack_f16x2(S[c8 + 6], S[c8 + 7]));
        }
        // Output row t = tid.
        {
            float y[BV];
            tmem_ld32(tmem + lane_off + (uint32_t)BV, y);
            tmem_ld_wait();
            const int t = tid;
            const int rows = len - j * BT < BT ? len - j * BT : BT;
            if (t < rows) {
                uint32_t w[BV / 2];
#pragma unroll
                for (int c8 = 0; c8 < BV; c8 += 8) {
                    const uint4 oi = *reinterpret_cast<const uint4*>(st + ST_OI + sw64_off(t, c8));
                    const float2 a0 = unpack_f16x2(oi.x), a1 = unpack_f16x2(oi.y), a2 = unpack_f16x2(oi.z),
                                 a3 = unpack_f16x2(oi.w);
                    w[c8 / 2 + 0] = pack_bf16x2(y[c8 + 0] + a0.x, y[c8 + 1] + a0.y);
                    w[c8 / 2 + 1] = pack_bf16x2(y[c8 + 2] + a1.x, y[c8 + 3] + a1.y);
                    w[c8 / 2 + 2] = pack_bf16x2(y[c8 + 4] + a2.x, y[c8 + 5] + a2.y);
                    w[c8 / 2 + 3] = pack_bf16x2(y[c8 + 6] + a3.x, y[c8 + 7] + a3.y);
                }
                uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)(bos + (long long)j * BT + t) * H + h) * VD +
                                                      vt * BV);
#pragma unroll
                for (int q4 = 0; q4 < BV / 8; ++q4)
                    dst[q4] = make_uint4(w[q4 * 4 + 0], w[q4 * 4 + 1], w[q4 * 4 + 2], w[q4 * 4 + 3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (*sFlag != 0) break;   // uniform after the barrier
        if (tid == 0 && j + 2 < nch) load_stage(p, chunk_slot(p, n, j + 2), h, vt, stage, s ? full1 : full0);
    }

    if (*sFlag != 0 && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
    if (p.ht != nullptr) {
#pragma unroll
        for (int j = 0; j < BV; ++j) p.ht[sbase_state + (size_t)(vt * BV + j) * KD + d] = S[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

cudaError_t launch_scan(const FwdParams& p, cudaStream_t stream) {
    const dim3 grid((unsigned)NVT, (unsigned)p.H, (unsigned)p.N);
    cudaError_t e = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_SMEM);
    if (e != cudaSuccess) return e;
    kda_scan_kernel<<<grid, SCAN_THREADS, SCAN_SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
