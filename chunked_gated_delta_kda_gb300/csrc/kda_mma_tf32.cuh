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

// Four 8 x 4 fp32 blocks (8 rows of 16 bytes each) into one register each:
// thread i gives the address of row i % 8 of block i / 8 and receives word
// (lane % 4) of row (lane / 4) of every block, which is the (g, t) position
// of an m16n8k8 TF32 fragment.  Row addresses must be 16-byte aligned.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const float* row_addr) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row_addr));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ uint32_t tf32_bits(uint32_t x) { return to_tf32(__uint_as_float(x)); }

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
    // row-major operands (A not transposed, B stored as [j][l]) come in by
    // ldmatrix, four fragment registers per instruction; the same 32-bit
    // words as the element loads, rounded the same way
    const int lr = lane & 7, lm = lane >> 3;
#pragma unroll 2
    for (int k0 = 0; k0 < kd; k0 += 8) {
        uint32_t a[MI][4], b[4][2];
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
            const int r = i0 + 16 * mi + g;
            if (!TA) {
                // blocks: rows +0 / +8 (lm & 1), columns k0 / k0 + 4 (lm >> 1)
                ldsm_x4(a[mi], A + (i0 + 16 * mi + 8 * (lm & 1) + lr) * MMA_LD + k0 + 4 * (lm >> 1));
#pragma unroll
                for (int e = 0; e < 4; ++e) a[mi][e] = tf32_bits(a[mi][e]);
            } else {
                a[mi][0] = to_tf32(opA(r, k0 + t));
                a[mi][1] = to_tf32(opA(r + 8, k0 + t));
                a[mi][2] = to_tf32(opA(r, k0 + t + 4));
                a[mi][3] = to_tf32(opA(r + 8, k0 + t + 4));
            }
        }
        if (TB) {
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                // blocks: columns k0 / k0 + 4 (lm & 1) of n-tiles 2 np / 2 np + 1 (lm >> 1)
                uint32_t q[4];
                ldsm_x4(q, B + (j0 + 8 * (2 * np + (lm >> 1)) + lr) * MMA_LD + k0 + 4 * (lm & 1));
                b[2 * np][0] = tf32_bits(q[0]);
                b[2 * np][1] = tf32_bits(q[1]);
                b[2 * np + 1][0] = tf32_bits(q[2]);
                b[2 * np + 1][1] = tf32_bits(q[3]);
            }
        } else {
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) {
                const int c = j0 + 8 * nj + g;
                b[nj][0] = to_tf32(opB(k0 + t, c));
                b[nj][1] = to_tf32(opB(k0 + t + 4, c));
            }
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi)
#pragma unroll
            for (int nj = 0; nj < 4; ++nj) mma_tf32(acc[mi][nj], a[mi], b[nj]);
    }
}

}  // namespace kda
