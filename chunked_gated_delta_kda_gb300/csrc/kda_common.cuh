// Shared definitions for the chunked KDA forward kernels: sizes, the per-chunk
// workspace tile layout, the chunk-slot map for fixed-length and varlen
// packing, and the device status word.
//
// Method (page "PyPTO-Gym chunk_kda operator: an NPU forward of chunked gated
// delta-rule linear attention", section "算法原理", steps M1-M4): split each
// sequence into chunks of BT = 128 tokens; inside a chunk build the gated
// k-k matrix A and the q-k matrix A2, invert (I + A), form the WY projections
// w and u, then walk the chunks in order carrying the K x V state S.
//
// This implementation re-associates step M4 exactly (no approximation):
//   v_new = u - w S,  o = qg S + A2 v_new,  S' = D S + kg^T v_new
// becomes
//   S' = D S + N S + Bc   with N = -kg^T w (K x K), Bc = kg^T u (K x V)
//   o  = Qe S + Oi        with Qe = qg - A2 w (BT x K), Oi = A2 u (BT x V)
// where qg = (scale q) * exp(G), kg = k * exp(G_last - G), D = diag(exp(G_last)).
// Everything except the S recurrence is chunk-parallel (the "prep" kernel);
// the recurrence is one K x K by K x V product per chunk (the "scan" kernel).
#pragma once

#include <cstdint>

namespace kda {

constexpr int BT = 128;   // chunk length (tokens)
constexpr int KD = 128;   // key / query head dimension
constexpr int VD = 128;   // value head dimension
constexpr int BV = 32;    // value-dimension tile of one scan CTA
constexpr int NVT = VD / BV;

// ---------------------------------------------------------------------------
// Per-(slot, head) workspace tile, written by the prep kernel and read by the
// scan kernel with 1-D bulk copies.  Each piece is stored byte-for-byte in the
// shared-memory layout the scan kernel's MMAs and threads expect.
//   Nm  : fp16 K x K, K-major 128B-swizzled (A operand: rows d_out, cols d_in)
//   Qe  : fp16 BT x K, K-major 128B-swizzled (A operand: rows t, cols d)
//   Bc  : fp16 [NVT][K][BV], each [K][BV] piece 64B-swizzled (row d)
//   Oi  : fp16 [NVT][BT][BV], each piece 64B-swizzled (row t)
//   Dg  : fp32 [K] = exp(G_last)
// ---------------------------------------------------------------------------
constexpr uint32_t TILE_NM = 0;
constexpr uint32_t TILE_QE = TILE_NM + KD * KD * 2;          // 32768
constexpr uint32_t TILE_BC = TILE_QE + BT * KD * 2;          // 65536
constexpr uint32_t BC_PIECE = KD * BV * 2;                   // 8192
constexpr uint32_t TILE_OI = TILE_BC + NVT * BC_PIECE;       // 98304
constexpr uint32_t OI_PIECE = BT * BV * 2;                   // 8192
constexpr uint32_t TILE_DG = TILE_OI + NVT * OI_PIECE;       // 131072
constexpr uint32_t TILE_BYTES = TILE_DG + KD * 4;            // 131584

// Workspace header: word 0 = device status bits, word 1 = number of entries
// in the wide-range work list, then (from byte 256) the list itself (one
// int32 work-item id per (chunk slot, head) at most), then the tiles.  The
// first 16 bytes are cleared at the start of every call.
constexpr uint32_t STATUS_BAD_CU = 1u;
constexpr uint32_t STATUS_TIMEOUT = 2u;
constexpr uint32_t STATUS_BAD_INDEX = 4u;   // token-by-token kernel: a state slot out of range
constexpr uint32_t WS_HEADER = 256;
constexpr uint32_t WS_CLEAR = 16;

// ---- warp helpers of the token-by-token kernels ----

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// All-reduce eight per-lane partial sums over the warp: a reduce-scatter by
// halving (xor 16, 8, 4: each step keeps half of the rows and adds the
// partner's half), a butterfly over the last two lane bits, then a gather of
// the eight totals.  17 shuffles instead of 40.
__device__ __forceinline__ void warp_sum8(float (&a)[8], int lane) {
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = h16 ? a[j] : a[j + 4];
        const float keep = h16 ? a[j + 4] : a[j];
        b[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = h8 ? b[j] : b[j + 2];
        const float keep = h8 ? b[j + 2] : b[j];
        c[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float d;
    {
        const float send = h4 ? c[0] : c[1];
        const float keep = h4 ? c[1] : c[0];
        d = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    // lane holds the total of row 4*h16 + 2*h8 + h4; fetch every row's total
#pragma unroll
    for (int r = 0; r < 8; ++r)
        a[r] = __shfl_sync(0xffffffffu, d, ((r >> 2) << 4) | (((r >> 1) & 1) << 3) | ((r & 1) << 2));
}

__device__ __forceinline__ void load4_bf16(const uint16_t* p, float (&x)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
}

// Bytes before the tiles for a workspace holding `items` (slot, head) tiles.
__host__ __device__ constexpr unsigned long long ws_tiles_offset(unsigned long long items) {
    return WS_HEADER + ((items * 4ull + 255ull) / 256ull) * 256ull;
}

// Poll limit for mbarrier waits (MMA / bulk-copy completion inside one CTA),
// used when FwdParams::wait_limit is 0.  A wait on another role of the same
// CTA gives up after the limit, sets the CTA's failure flag and returns;
// every later wait of that CTA then returns at once, so a stalled CTA leaves
// within one limit.  Before it frees its TMEM or shared memory a CTA waits
// (with DRAIN_LIMIT, never skipped) for the copies and products it issued
// itself: those complete on their own.
constexpr uint32_t WAIT_LIMIT = 1u << 24;
constexpr uint32_t DRAIN_LIMIT = 1u << 24;

// FwdParams::debug bits (failure-detection tests only; see kda_debug_set)
constexpr uint32_t DEBUG_DROP_SCAN_LOAD = 1u;   // scan: unit (0, 0), V tile 0 never loads chunk 1's stage

struct FwdParams {
    const uint16_t* q;      // bf16 [B*T, H, K]
    const uint16_t* k;      // bf16 [B*T, H, K]
    const uint16_t* v;      // bf16 [B*T, H, V]
    const float* g;         // fp32 [B*T, H, K]
    const float* beta;      // fp32 [B*T, H]
    const float* h0;        // fp32 [N, H, V, K] or null
    const int32_t* cu;      // int32 [N+1] or null (fixed length)
    uint16_t* o;            // bf16 [B*T, H, V]
    float* ht;              // fp32 [N, H, V, K] or null
    uint8_t* tiles;         // workspace tiles, [nslots][H][TILE_BYTES]
    uint32_t* status;       // workspace status word
    uint32_t* wide_count;   // number of work items queued for the wide-range path
    int32_t* wide_list;     // their ids (slot * H + head)
    uint32_t* exact_flags;  // [N][H]: 1 where a chunk exceeded the exact factoring range
    float* ckpt;            // scan: fp32 [nslots][H][K][V], the state entering each chunk, or null
    float scale;
    int T;                  // per-sequence length (fixed) or packed length (varlen)
    int H;
    int N;
    int NT;                 // chunks per sequence (fixed length), else 0
    int nslots;             // number of chunk slots the workspace holds
    uint32_t wait_limit;    // poll limit of the bounded waits (0: WAIT_LIMIT)
    uint32_t debug;         // DEBUG_* bits (0 in normal use)
};

__device__ __forceinline__ uint32_t wait_limit_of(const FwdParams& p) {
    return p.wait_limit != 0u ? p.wait_limit : WAIT_LIMIT;
}

// A chunk: sequence n, chunk j inside it, first token (packed index), rows.
struct ChunkRef {
    int n;
    int j;
    long long tok0;
    int len;
    int slot;
};

__device__ __forceinline__ int cdiv128(int x) { return (x + BT - 1) / BT; }

// Slot of chunk 0 of sequence n (varlen): floor(cu[n]/BT) + n.  Strictly
// increasing in n and injective over (n, j) for j < ceil(len_n / BT), so a
// workspace of floor(T/BT) + N + 1 slots per head holds every chunk.
__device__ __forceinline__ int varlen_base(const int32_t* cu, int n) { return cu[n] / BT + n; }

// Sequence bounds with validation: returns false (and flags the status word)
// if cu is not a valid non-decreasing offset list into [0, T].
__device__ __forceinline__ bool seq_bounds(const FwdParams& p, int n, long long& bos, int& len) {
    if (p.cu == nullptr) {
        bos = (long long)n * p.T;
        len = p.T;
        return true;
    }
    const int a = p.cu[n];
    const int b = p.cu[n + 1];
    if (a < 0 || b < a || b > p.T || (n == 0 && a != 0) || (n == p.N - 1 && b != p.T)) {
        atomicOr(p.status, STATUS_BAD_CU);
        return false;
    }
    bos = a;
    len = b - a;
    return true;
}

__device__ __forceinline__ int chunk_slot(const FwdParams& p, int n, int j) {
    return p.cu == nullptr ? n * p.NT + j : varlen_base(p.cu, n) + j;
}

// Map a slot back to its chunk (prep kernel).  Returns false for slots that
// hold no chunk (gaps in the varlen map, or slots past the end).
__device__ __forceinline__ bool slot_chunk(const FwdParams& p, int slot, ChunkRef& c) {
    int n, j;
    if (p.cu == nullptr) {
        if (slot >= p.N * p.NT) return false;
        n = slot / p.NT;
        j = slot % p.NT;
    } else {
        // largest n in [0, N) with base(n) <= slot
        int lo = 0, hi = p.N - 1;
        if (p.N <= 0 || varlen_base(p.cu, 0) > slot) return false;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (varlen_base(p.cu, mid) <= slot) lo = mid;
            else hi = mid - 1;
        }
        n = lo;
        j = slot - varlen_base(p.cu, n);
    }
    long long bos;
    int len;
    if (!seq_bounds(p, n, bos, len)) return false;
    if (j * BT >= len) return false;
    c.n = n;
    c.j = j;
    c.tok0 = bos + (long long)j * BT;
    c.len = len - j * BT < BT ? len - j * BT : BT;
    c.slot = slot;
    return true;
}

__device__ __forceinline__ uint8_t* tile_ptr(const FwdParams& p, int slot, int h) {
    return p.tiles + ((size_t)slot * p.H + h) * TILE_BYTES;
}

}  // namespace kda
