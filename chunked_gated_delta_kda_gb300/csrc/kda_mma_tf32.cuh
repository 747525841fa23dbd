// Warp-level TF32 tensor-core products (mma.sync m16n8k8, fp32 accumulation)
// on fp32 matrices in shared memory with rows of MMA_LD floats (128 + 4 of
// padding, so that the fragment loads of a warp hit distinct banks).
#pragma once

#include <cstdint>

namespace kda {

constexpr int MMA_LD = 132;

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc (a (16 MI) x 32 tile at rows i0, cols j0) += opA(i0.., 0..kd) opB(0..kd, j0..)
// with opA(i, l) = TA ? A[l][i] : A[i][l] and opB(l, j) = TB ? B[j][l] : B[l][j],
// shared buffers of row length MMA_LD.  Fragment layouts of m16n8k8
// (g = lane / 4, t = lane % 4): A: (g, t) (g+8, t) (g, t+4) (g+8, t+4);
// B: (t, g) (t+4, g); D: (g, 2t) (g, 2t+1) (g+8, 2t) (g+8, 2t+1).
template <bool TA, bool TB, int MI>
__device__ __forceinline__ void tile_mm(const float* A, const float* B, int i0, int j0, int kd, int lane,
                                        float (&acc)[MI][4][4]) {
    const int g = lane >> 2, t = lane & 3;
    auto opA = [&](int i, int l) { return TA ? A[l * MMA_LD + i] : A[i * MMA_LD + l]; };
    auto opB = [&](int l, int j) { return TB ? B[j * MMA_LD + l] : B[l * MMA_LD + j]; };
#pragma unroll 2
    for (int k0 = 0; k0 < kd; k0 += 8) {
        uint32_t a[MI][4], b[4][2];
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
            const int r = i0 + 16 * mi + g;
            a[mi][0] = to_tf32(opA(r, k0 + t));
            a[mi][1] = to_tf32(opA(r + 8, k0 + t));
            a[mi][2] = to_tf32(opA(r, k0 + t + 4));
            a[mi][3] = to_tf32(opA(r + 8, k0 + t + 4));
        }
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
            const int c = j0 + 8 * nj + g;
            b[nj][0] = to_tf32(opB(k0 + t, c));
            b[nj][1] = to_tf32(opB(k0 + t + 4, c));
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi)
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) mma_tf32(acc[mi][nj], a[mi], b[nj]);
    }
}

}  // namespace kda
