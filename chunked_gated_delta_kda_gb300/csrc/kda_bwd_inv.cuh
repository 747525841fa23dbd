// The unit lower-triangular inverse of the chunked backward, on a 128 x 128
// fp32 matrix in shared memory with rows of MMA_LD floats, by a CTA of 16
// warps: 16 x 16 diagonal blocks by forward substitution (fp32), then merges
// 16 -> 32 -> 64 -> 128 with inv([[A, 0], [C, D]]) = [[A^-1, 0], [-D^-1 C A^-1, D^-1]]
// on the TF32 tensor cores (mma.sync).
#pragma once

#include "kda_common.cuh"
#include "kda_mma_tf32.cuh"

namespace kda {

constexpr int INV_WARPS = 16;

// 16 x 16 tiles for the inverse's merges: acc (m16 x n16) += opA opB over kd.
template <bool TA, bool TB>
__device__ __forceinline__ void tile16_mm(const float* A, const float* B, int kd, int lane, float (&acc)[2][4]) {
    const int g = lane >> 2, t = lane & 3;
    for (int k0 = 0; k0 < kd; k0 += 8) {
        uint32_t a[4], b[2][2];
        auto opA = [&](int i, int l) { return TA ? A[l * MMA_LD + i] : A[i * MMA_LD + l]; };
        auto opB = [&](int l, int j) { return TB ? B[j * MMA_LD + l] : B[l * MMA_LD + j]; };
        a[0] = to_tf32(opA(g, k0 + t));
        a[1] = to_tf32(opA(g + 8, k0 + t));
        a[2] = to_tf32(opA(g, k0 + t + 4));
        a[3] = to_tf32(opA(g + 8, k0 + t + 4));
#pragma unroll
        for (int nj = 0; nj < 2; ++nj) {
            b[nj][0] = to_tf32(opB(k0 + t, 8 * nj + g));
            b[nj][1] = to_tf32(opB(k0 + t + 4, 8 * nj + g));
        }
        mma_tf32(acc[0], a, b[0]);
        mma_tf32(acc[1], a, b[1]);
    }
}

// In-place inverse of the unit lower-triangular 128 x 128 matrix in L (row length MMA_LD).
// The strictly upper part must be zero on entry; it stays zero.
static __device__ void invert_unit_lower(float* L, int warp, int lane, int tid) {
    // level 0: the eight 16 x 16 diagonal blocks, one warp each, lane j = column j
    if (warp < 8 && lane < 16) {
        float* blk = L + (16 * warp) * MMA_LD + 16 * warp;
        const int j = lane;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m < i) s = fmaf(blk[i * MMA_LD + m], x[m], s);
            if (i > j) x[i] = -s;
        }
        __syncwarp(0xffffu);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (i >= j) blk[i * MMA_LD + j] = x[i];
    }
    __syncthreads();
    // merges: for block size s, pairs at a = 2 p s: C = L[a+s.., a..] -> -D^-1 C A^-1
    for (int s = 16; s < BT; s *= 2) {
        const int pairs = BT / (2 * s);
        const int tiles = pairs * (s / 16) * (s / 16);   // 16 x 16 output tiles over all pairs
        // T = C A^-1 (into registers), then written over C
        float acc[2][2][4];
        int nt = 0;
        for (int tI = warp; tI < tiles; tI += INV_WARPS, ++nt) {
            const int per = (s / 16) * (s / 16);
            const int pr = tI / per, rem = tI % per;
            const int a = 2 * pr * s, ti = rem / (s / 16), tj = rem % (s / 16);
            float(&c)[2][4] = acc[nt];
            for (int u = 0; u < 2; ++u) c[u][0] = c[u][1] = c[u][2] = c[u][3] = 0.f;
            tile16_mm<false, false>(L + (a + s + 16 * ti) * MMA_LD + a, L + a * MMA_LD + a + 16 * tj, s, lane, c);
        }
        __syncthreads();
        nt = 0;
        for (int tI = warp; tI < tiles; tI += INV_WARPS, ++nt) {
            const int per = (s / 16) * (s / 16);
            const int pr = tI / per, rem = tI % per;
            const int a = 2 * pr * s, ti = rem / (s / 16), tj = rem % (s / 16);
            const int g = lane >> 2, t = lane & 3;
            float* dst = L + (a + s + 16 * ti) * MMA_LD + a + 16 * tj;
            for (int u = 0; u < 2; ++u) {
                dst[g * MMA_LD + 8 * u + 2 * t] = acc[nt][u][0];
                dst[g * MMA_LD + 8 * u + 2 * t + 1] = acc[nt][u][1];
                dst[(g + 8) * MMA_LD + 8 * u + 2 * t] = acc[nt][u][2];
                dst[(g + 8) * MMA_LD + 8 * u + 2 * t + 1] = acc[nt][u][3];
            }
        }
        __syncthreads();
        // C' = -D^-1 T
        nt = 0;
        for (int tI = warp; tI < tiles; tI += INV_WARPS, ++nt) {
            const int per = (s / 16) * (s / 16);
            const int pr = tI / per, rem = tI % per;
            const int a = 2 * pr * s, ti = rem / (s / 16), tj = rem % (s / 16);
            float(&c)[2][4] = acc[nt];
            for (int u = 0; u < 2; ++u) c[u][0] = c[u][1] = c[u][2] = c[u][3] = 0.f;
            tile16_mm<false, false>(L + (a + s + 16 * ti) * MMA_LD + a + s, L + (a + s) * MMA_LD + a + 16 * tj, s, lane, c);
        }
        __syncthreads();
        nt = 0;
        for (int tI = warp; tI < tiles; tI += INV_WARPS, ++nt) {
            const int per = (s / 16) * (s / 16);
            const int pr = tI / per, rem = tI % per;
            const int a = 2 * pr * s, ti = rem / (s / 16), tj = rem % (s / 16);
            const int g = lane >> 2, t = lane & 3;
            float* dst = L + (a + s + 16 * ti) * MMA_LD + a + 16 * tj;
            for (int u = 0; u < 2; ++u) {
                dst[g * MMA_LD + 8 * u + 2 * t] = -acc[nt][u][0];
                dst[g * MMA_LD + 8 * u + 2 * t + 1] = -acc[nt][u][1];
                dst[(g + 8) * MMA_LD + 8 * u + 2 * t] = -acc[nt][u][2];
                dst[(g + 8) * MMA_LD + 8 * u + 2 * t + 1] = -acc[nt][u][3];
            }
        }
        __syncthreads();
    }
    (void)tid;
}

}  // namespace kda
