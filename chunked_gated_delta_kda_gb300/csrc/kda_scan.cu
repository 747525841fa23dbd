// Sequential half of the chunked KDA forward ("scan"): for one (sequence,
// head, 32-wide value tile) it walks the chunks in order carrying the state
// S (K x 32, fp32, one row per thread) and produces the output rows:
//   S' = Dg * S + Nm S + Bc,     o = Qe S + Oi
// With o null it runs the state recurrence alone (the backward runs it on
// transposed tiles in reverse chunk order to carry the state gradient), and
// with ckpt set it also stores the fp32 state entering every chunk.
// which is step M4 of the page "PyPTO-Gym chunk_kda operator: an NPU forward
// of chunked gated delta-rule linear attention" (section "算法原理") in the
// exact re-associated form set out in kda_common.cuh.  The initial and final
// states use the page's [N, H, V, K] layout (section "算子签名与 I/O 规格"),
// i.e. the transpose of the K x V state; the transpose happens here.
//
// GB300 mapping.  352 threads in five roles, handing work to each other
// through mbarriers so that no role waits on another's latency:
//   warps 0-3  state:  thread i owns row d = i of S (fp32, registers); per
//              chunk it reads Nm S from TMEM, applies S' = Dg S + Nm S + Bc
//              and writes the fp16 copy of S' the next chunk's MMAs read;
//   warps 4-7  output: thread i owns row t = i; reads Qe S from one of two
//              TMEM buffers, adds Oi, rounds to bf16 and stores o;
//   warp 8     MMA issue: the Nm S product of chunk j (the critical chain),
//              then the Qe S product of chunk j - 1, which runs while the
//              state warps update chunk j;
//   warp 9     loads of the critical-path stages, two chunks ahead;
//   warp 10    loads of the output tiles (Qe, Oi).
// The critical-path tiles (Nm, Bc piece, Dg) are double-buffered in stages
// that free as soon as the state update is done; Qe has its own two-slot
// ring (its product lags one chunk), Oi a four-slot ring, and the fp16 state
// copy three buffers (chunk j's copy is read by Qe S one chunk later).
#include "kda_common.cuh"
#include "sm100_ptx.cuh"

namespace kda {

namespace {

constexpr int SCAN_THREADS = 352;
// the loaders also prefetch the tiles this many chunks ahead into L2, so
// that the stage loads (two chunks ahead) find them there rather than in DRAM
constexpr int PF_AHEAD = 4;
// stage: Nm | Bc piece | Dg
constexpr uint32_t ST_NM = 0;
constexpr uint32_t ST_BC = 32768;
constexpr uint32_t ST_DG = 40960;
constexpr uint32_t ST_BYTES = 41472;          // bytes loaded per stage
constexpr uint32_t ST_STRIDE = 41984;         // 1024-aligned stage stride
constexpr uint32_t S_QE = 2 * ST_STRIDE;      // Qe ring: 2 x 32 KB
constexpr uint32_t S_OI = S_QE + 2 * 32768;   // Oi ring: 4 x 8 KB
constexpr uint32_t S_S16 = S_OI + 4 * OI_PIECE;   // fp16 state copies: 3 x [K][32] 64B-swizzled
constexpr uint32_t S_BAR = S_S16 + 3 * 8192;
// barrier offsets (8 bytes each)
constexpr uint32_t B_FULL = 0, B_QFULL = 16, B_OIFULL = 32, B_OIFREE = 64, B_MMAS = 96, B_MMAO = 104,
                   B_OFREE = 120, B_S16 = 136, B_SFREE = 144, B_DRAIN = 160;
constexpr uint32_t S_TMEM = S_BAR + 192;
constexpr uint32_t S_FLAG = S_TMEM + 4;
constexpr uint32_t SCAN_SMEM = S_BAR + 256 + 1024;

__device__ __forceinline__ void load_stage(const FwdParams& p, int slot, int h, int vt, uint32_t dst,
                                           uint32_t bar) {
    const uint8_t* src = tile_ptr(p, slot, h);
    mbar_arrive_expect_tx(bar, ST_BYTES);
    bulk_g2s(dst + ST_NM, src + TILE_NM, KD * KD * 2, bar);
    bulk_g2s(dst + ST_BC, src + TILE_BC + vt * BC_PIECE, BC_PIECE, bar);
    bulk_g2s(dst + ST_DG, src + TILE_DG, KD * 4, bar);
}

__device__ __forceinline__ void load_piece(const uint8_t* src, uint32_t bytes, uint32_t dst, uint32_t bar) {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(dst, src, bytes, bar);
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
__device__ __forceinline__ void bar_sync_named(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
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
    const int lane = tid & 31;
    const int row = tid & 127;                      // state row d, or output row t

    long long bos;
    int len;
    if (!seq_bounds(p, n, bos, len)) return;        // uniform
    const int nch = (len + BT - 1) / BT;

    const uint32_t bars = sbase + S_BAR;
    auto full = [&](int s) { return bars + B_FULL + 8u * (uint32_t)s; };
    auto qfull = [&](int s) { return bars + B_QFULL + 8u * (uint32_t)s; };
    auto oifull = [&](int r) { return bars + B_OIFULL + 8u * (uint32_t)r; };
    auto oifree = [&](int r) { return bars + B_OIFREE + 8u * (uint32_t)r; };
    auto mmao = [&](int b) { return bars + B_MMAO + 8u * (uint32_t)b; };
    auto ofree = [&](int b) { return bars + B_OFREE + 8u * (uint32_t)b; };
    auto sfree = [&](int s) { return bars + B_SFREE + 8u * (uint32_t)s; };
    auto s16buf = [&](int j) { return S_S16 + (uint32_t)(j % 3) * 8192u; };
    const uint32_t mmas = bars + B_MMAS, s16rdy = bars + B_S16, drain = bars + B_DRAIN;
    volatile uint32_t* sFlag = reinterpret_cast<volatile uint32_t*>(sm + S_FLAG);
    if (warp == 0) {
        tmem_alloc(sbase + S_TMEM, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(full(i), 1);
            mbar_init(qfull(i), 1);
            mbar_init(mmao(i), 1);
            mbar_init(ofree(i), 1);
            mbar_init(sfree(i), 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(oifull(i), 1);
            mbar_init(oifree(i), 1);
        }
        mbar_init(mmas, 1);
        mbar_init(s16rdy, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
        *sFlag = 0;
    }

    // State rows: state thread d holds S[d][vt*32 .. vt*32+31] (fp32).
    float S[BV];
    const size_t sbase_state = ((size_t)n * H + h) * VD * KD;   // [N,H,V,K] slab
    if (warp < 4) {
        if (p.h0 != nullptr) {
#pragma unroll
            for (int j = 0; j < BV; ++j) S[j] = __ldg(p.h0 + sbase_state + (size_t)(vt * BV + j) * KD + row);
        } else {
#pragma unroll
            for (int j = 0; j < BV; ++j) S[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < BV; j += 8)
            *reinterpret_cast<uint4*>(sm + s16buf(0) + sw64_off(row, j)) =
                make_uint4(pack_f16x2(S[j], S[j + 1]), pack_f16x2(S[j + 2], S[j + 3]),
                           pack_f16x2(S[j + 4], S[j + 5]), pack_f16x2(S[j + 6], S[j + 7]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + S_TMEM);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    // A wait on another role.  When one runs out the CTA's flag is set and
    // the role leaves its loop at once (one decision per role, taken by vote
    // so that the role's barriers still match); a role waiting on a role that
    // has left runs out in its turn, so the CTA is done within about two
    // limits.  (Checking the flag before every wait instead cost ~10% here.)
    const uint32_t wlim = wait_limit_of(p);
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity, wlim)) return true;
        *sFlag = 1;
        return false;
    };

    if (warp < 4) {
        // ------------------------------------------------------------------
        // State: S' = Dg S + Nm S + Bc, row d = tid.
        // ------------------------------------------------------------------
        bool alive = true;
        for (int j = 0; j < nch; ++j) {
            const int s = j & 1;
            if (p.ckpt != nullptr) {   // the state entering chunk j, row d, [K][V] layout
                float4* ck = reinterpret_cast<float4*>(p.ckpt + (((size_t)chunk_slot(p, n, j) * H + h) * KD + row) * VD +
                                                       vt * BV);
#pragma unroll
                for (int c4 = 0; c4 < BV / 4; ++c4)
                    ck[c4] = make_float4(S[4 * c4], S[4 * c4 + 1], S[4 * c4 + 2], S[4 * c4 + 3]);
            }
            bool ok = wait(full(s), (uint32_t)(j >> 1) & 1u);   // Bc / Dg of this chunk have landed
            ok = ok && wait(mmas, (uint32_t)j & 1u);
            ok = __all_sync(0xffffffffu, ok);               // warp-uniform before tcgen05.ld
            tc_fence_after();
            if (ok) {
            const uint8_t* st = sm + (size_t)s * ST_STRIDE;
            float x[BV];
            tmem_ld32(tmem + lane_off, x);
            tmem_ld_wait();
            const float Dd = *reinterpret_cast<const float*>(st + ST_DG + row * 4);
#pragma unroll
            for (int c8 = 0; c8 < BV; c8 += 8) {
                const uint4 bc = *reinterpret_cast<const uint4*>(st + ST_BC + sw64_off(row, c8));
                const float2 b0 = unpack_f16x2(bc.x), b1 = unpack_f16x2(bc.y), b2 = unpack_f16x2(bc.z),
                             b3 = unpack_f16x2(bc.w);
                S[c8 + 0] = fmaf(Dd, S[c8 + 0], x[c8 + 0] + b0.x);
                S[c8 + 1] = fmaf(Dd, S[c8 + 1], x[c8 + 1] + b0.y);
                S[c8 + 2] = fmaf(Dd, S[c8 + 2], x[c8 + 2] + b1.x);
                S[c8 + 3] = fmaf(Dd, S[c8 + 3], x[c8 + 3] + b1.y);
                S[c8 + 4] = fmaf(Dd, S[c8 + 4], x[c8 + 4] + b2.x);
                S[c8 + 5] = fmaf(Dd, S[c8 + 5], x[c8 + 5] + b2.y);
                S[c8 + 6] = fmaf(Dd, S[c8 + 6], x[c8 + 6] + b3.x);
                S[c8 + 7] = fmaf(Dd, S[c8 + 7], x[c8 + 7] + b3.y);
            }
            // the copy for chunk j + 1 goes to buffer (j + 1) % 3, last read
            // by the products of chunk j - 2: Nm S(j - 2) and Qe S(j - 2),
            // both issued before Nm S(j), whose commit we waited for
            uint8_t* s16 = sm + s16buf(j + 1);
#pragma unroll
            for (int c8 = 0; c8 < BV; c8 += 8)
                *reinterpret_cast<uint4*>(s16 + sw64_off(row, c8)) =
                    make_uint4(pack_f16x2(S[c8], S[c8 + 1]), pack_f16x2(S[c8 + 2], S[c8 + 3]),
                               pack_f16x2(S[c8 + 4], S[c8 + 5]), pack_f16x2(S[c8 + 6], S[c8 + 7]));
            }
            fence_async_smem();
            tc_fence_before();
            if (!bar_and_named(1, 128, ok)) {
                alive = false;
                break;
            }
            if (tid == 0) {
                mbar_arrive(s16rdy);      // next chunk's MMAs may start
                mbar_arrive(sfree(s));    // Nm / Bc / Dg of stage s are consumed
            }
        }
        if (alive && p.ht != nullptr) {
#pragma unroll
            for (int j = 0; j < BV; ++j) p.ht[sbase_state + (size_t)(vt * BV + j) * KD + row] = S[j];
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------------
        // Output: o rows of chunk j from TMEM buffer j & 1 plus Oi (none
        // when o is null: a state-only pass).
        // ------------------------------------------------------------------
        for (int j = 0; j < (p.o != nullptr ? nch : 0); ++j) {
            const int b = j & 1, r = j & 3;
            bool ok = wait(mmao(b), (uint32_t)(j >> 1) & 1u);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            float y[BV];
            if (ok) {
                tmem_ld32(tmem + lane_off + 32u + 32u * (uint32_t)b, y);
                tmem_ld_wait();
            }
            tc_fence_before();
            if (!bar_and_named(2, 128, ok)) break;
            if (tid == 128) mbar_arrive(ofree(b));
            ok = wait(oifull(r), (uint32_t)(j >> 2) & 1u);
            const int rows = len - j * BT < BT ? len - j * BT : BT;
            if (ok && row < rows) {
                const uint8_t* oi_s = sm + S_OI + (uint32_t)r * OI_PIECE;
                uint32_t w[BV / 2];
#pragma unroll
                for (int c8 = 0; c8 < BV; c8 += 8) {
                    const uint4 oi = *reinterpret_cast<const uint4*>(oi_s + sw64_off(row, c8));
                    const float2 a0 = unpack_f16x2(oi.x), a1 = unpack_f16x2(oi.y), a2 = unpack_f16x2(oi.z),
                                 a3 = unpack_f16x2(oi.w);
                    w[c8 / 2 + 0] = pack_bf16x2(y[c8 + 0] + a0.x, y[c8 + 1] + a0.y);
                    w[c8 / 2 + 1] = pack_bf16x2(y[c8 + 2] + a1.x, y[c8 + 3] + a1.y);
                    w[c8 / 2 + 2] = pack_bf16x2(y[c8 + 4] + a2.x, y[c8 + 5] + a2.y);
                    w[c8 / 2 + 3] = pack_bf16x2(y[c8 + 6] + a3.x, y[c8 + 7] + a3.y);
                }
                uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)(bos + (long long)j * BT + row) * H + h) * VD +
                                                      vt * BV);
#pragma unroll
                for (int q4 = 0; q4 < BV / 8; ++q4)
                    dst[q4] = make_uint4(w[q4 * 4 + 0], w[q4 * 4 + 1], w[q4 * 4 + 2], w[q4 * 4 + 3]);
            }
            if (!bar_and_named(2, 128, ok)) break;
            if (tid == 128) mbar_arrive(oifree(r));
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------------
        // MMA issue (the whole warp computes the operands, one elected lane
        // issues): Nm S(j), then Qe S(j - 1).
        // ------------------------------------------------------------------
        {
            const uint32_t id = idesc_f16(T_F16, 128, BV, false, true);
            // per k-step only the start-address field of these advances
            const uint64_t a_nm0 = smem_desc(sbase + ST_NM, 16u, 1024u, SW_128B);
            const uint64_t a_nm1 = smem_desc(sbase + ST_STRIDE + ST_NM, 16u, 1024u, SW_128B);
            const uint64_t a_qe0 = smem_desc(sbase + S_QE, 16u, 1024u, SW_128B);
            const uint64_t a_qe1 = smem_desc(sbase + S_QE + 32768u, 16u, 1024u, SW_128B);
            for (int j = 0; j <= nch; ++j) {
                if (j < nch) {
                    const int s = j & 1;
                    bool ok = wait(full(s), (uint32_t)(j >> 1) & 1u);
                    if (j >= 1) ok = ok && wait(s16rdy, (uint32_t)(j - 1) & 1u);
                    // reconverged and warp-uniform before elect.sync
                    if (!__all_sync(0xffffffffu, ok)) break;
                    tc_fence_after();
                    const uint64_t a_nm = s ? a_nm1 : a_nm0;
                    const uint64_t b_s = smem_desc(sbase + s16buf(j), 512u, 512u, SW_64B);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // critical chain: Nm S -> cols [0,32)
                        mma_f16_warp(tmem, a_nm + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2), b_s + (uint64_t)(ks * 64),
                                id, ks > 0);
                    mma_commit_warp(mmas);
                }
                if (j >= 1 && p.o != nullptr) {
                    const int c = j - 1, b = c & 1;
                    bool ok = wait(qfull(b), (uint32_t)(c >> 1) & 1u);
                    if (c >= 2) ok = ok && wait(ofree(b), (uint32_t)((c - 2) >> 1) & 1u);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    tc_fence_after();
                    const uint64_t a_qe = b ? a_qe1 : a_qe0;
                    const uint64_t b_s = smem_desc(sbase + s16buf(c), 512u, 512u, SW_64B);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // output product Qe S(c) -> buffer b
                        mma_f16_warp(tmem + 32u + 32u * (uint32_t)b, a_qe + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2),
                                b_s + (uint64_t)(ks * 64), id, ks > 0);
                    mma_commit_warp(mmao(b));
                }
            }
            // every product issued above has completed before TMEM is freed
            mma_commit_warp(drain);
            mbar_wait(drain, 0, DRAIN_LIMIT);
        }
    } else {
        // ------------------------------------------------------------------
        // Loads, from two warps so that the critical-path tiles never queue
        // behind the lagging output product (two spinning lanes of one warp
        // would serialise):
        //   warp 9:  the stage (Nm, Bc, Dg) two chunks ahead, once the state
        //            warps are done with it;
        //   warp 10: Qe once its product of two chunks back has completed,
        //            Oi once its slot has been read.
        // ------------------------------------------------------------------
        // Before the CTA exits each loader waits for the last copy it issued
        // into every buffer slot (copies complete on their own); chunk c's
        // copy completes phase c / (ring size) of its slot's barrier.  The
        // last chunk per slot is kept in scalars (an indexed array here goes
        // to local memory and slowed the scan by ~15%).
        if (warp == 9 && lane == 0) {
            int last0 = -1, last1 = -1;   // last chunk loaded into stage 0 / 1
            const bool drop = (p.debug & DEBUG_DROP_SCAN_LOAD) != 0u && n == 0 && h == 0 && vt == 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                if (c >= 2 && !wait(sfree(s), (uint32_t)((c - 2) >> 1) & 1u)) break;
                if (drop && c == 1) continue;   // failure-detection test: this stage never arrives
                load_stage(p, chunk_slot(p, n, c), h, vt, sbase + (uint32_t)s * ST_STRIDE, full(s));
                if (c + PF_AHEAD < nch) {   // the stage PF_AHEAD chunks on into L2
                    const uint8_t* pf = tile_ptr(p, chunk_slot(p, n, c + PF_AHEAD), h);
                    bulk_prefetch_l2(pf + TILE_NM, KD * KD * 2);
                    bulk_prefetch_l2(pf + TILE_BC + vt * BC_PIECE, BC_PIECE);
                    bulk_prefetch_l2(pf + TILE_DG, KD * 4);
                }
                if (s) last1 = c;
                else last0 = c;
            }
            if (last0 >= 0) mbar_wait(full(0), (uint32_t)(last0 >> 1) & 1u, DRAIN_LIMIT);
            if (last1 >= 0) mbar_wait(full(1), (uint32_t)(last1 >> 1) & 1u, DRAIN_LIMIT);
        } else if (warp == 10 && lane == 0 && p.o != nullptr) {
            int nq = 0, no = 0;           // chunks whose Qe / Oi copies were issued (in order)
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1, r = c & 3;
                const uint8_t* src = tile_ptr(p, chunk_slot(p, n, c), h);
                if (c >= 2 && !wait(mmao(s), (uint32_t)((c - 2) >> 1) & 1u)) break;
                load_piece(src + TILE_QE, BT * KD * 2, sbase + S_QE + (uint32_t)s * 32768u, qfull(s));
                nq = c + 1;
                if (c + PF_AHEAD < nch) {
                    const uint8_t* pf = tile_ptr(p, chunk_slot(p, n, c + PF_AHEAD), h);
                    bulk_prefetch_l2(pf + TILE_QE, BT * KD * 2);
                    bulk_prefetch_l2(pf + TILE_OI + vt * OI_PIECE, OI_PIECE);
                }
                if (c >= 4 && !wait(oifree(r), (uint32_t)((c - 4) >> 2) & 1u)) break;
                load_piece(src + TILE_OI + vt * OI_PIECE, OI_PIECE, sbase + S_OI + (uint32_t)r * OI_PIECE, oifull(r));
                no = c + 1;
            }
            for (int c = nq - 2 < 0 ? 0 : nq - 2; c < nq; ++c)
                mbar_wait(qfull(c & 1), (uint32_t)(c >> 1) & 1u, DRAIN_LIMIT);
            for (int c = no - 4 < 0 ? 0 : no - 4; c < no; ++c)
                mbar_wait(oifull(c & 3), (uint32_t)(c >> 2) & 1u, DRAIN_LIMIT);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*sFlag != 0 && tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, 128);
}

cudaError_t launch_scan(const FwdParams& p, cudaStream_t stream) {
    const dim3 grid((unsigned)NVT, (unsigned)p.H, (unsigned)p.N);
    cudaError_t e = cudaFuncSetAttribute(kda_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SCAN_SMEM);
    if (e != cudaSuccess) return e;
    kda_scan_kernel<<<grid, SCAN_THREADS, SCAN_SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
