// Parameters shared by the backward kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime_api.h>

namespace kda {

struct BwdParams {
    const uint16_t* q;      // bf16 [B*T, H, K]
    const uint16_t* k;      // bf16 [B*T, H, K]
    const uint16_t* v;      // bf16 [B*T, H, V]
    const float* g;         // fp32 [B*T, H, K]
    const float* beta;      // fp32 [B*T, H]
    const float* h0;        // fp32 [N, H, V, K] or null
    const int32_t* cu;      // int32 [N+1] or null (fixed length)
    const uint16_t* dout;   // bf16 [B*T, H, V]: dL/do
    const float* dht;       // fp32 [N, H, V, K] or null: dL/dht
    float* dq;              // fp32 [B*T, H, K]
    float* dk;              // fp32 [B*T, H, K]
    float* dv;              // fp32 [B*T, H, V]
    float* dg;              // fp32 [B*T, H, K]
    float* dbeta;           // fp32 [B*T, H]
    float* dh0;             // fp32 [N, H, V, K] or null
    float* ckpt;            // token-by-token kernel: fp32 [nslots][H][V][K], state entering each chunk
    float* scratch;         // fp32 [ctas][BT][V][K]: states entering tokens of a chunk
    const float* ckpt_s;    // chunk kernel: fp32 [nslots][H][K][V], S entering each chunk (forward scan)
    const float* ckpt_d;    // chunk kernel: fp32 [nslots][H][K][V], dS at the end of the mirrored chunk
    uint32_t* tc_skip;      // [nslots * H]: 1 where the tensor-core kernel left the chunk to the per-token kernel
    uint32_t* status;
    float scale;
    int T, H, N;
    int NT;                 // chunks per sequence (fixed length), else 0
    int l2norm;
};

struct FwdParams;
cudaError_t launch_bwd_tiles(const FwdParams& fp, uint8_t* btiles, const uint16_t* dout, cudaStream_t stream);
cudaError_t launch_bwd_chunk(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream);
cudaError_t launch_bwd_tc(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream);
cudaError_t launch_bwd_umma(const BwdParams& p, const FwdParams& fp, int ctas, cudaStream_t stream);
cudaError_t launch_bwd_exact(const BwdParams& p, const uint32_t* only, int ctas, cudaStream_t stream);
cudaError_t launch_l2norm_bwd(const BwdParams& p, long long rows, cudaStream_t stream);

}  // namespace kda
