/*
 * kda.h -- C ABI of the chunked Kimi Delta Attention (KDA) forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (page "PyPTO-Gym chunk_kda operator: an NPU forward of chunked
 * gated delta-rule linear attention"):
 *   per sequence n and head h, with the K x V state S starting at h0[n,h]^T
 *   (or zero) and, for every token t in order,
 *       S <- diag(exp(g_t)) S                       (per-dimension gate decay)
 *       S <- S + beta_t k_t (v_t - S^T k_t)^T       (delta update)
 *       o_t = S^T (scale q_t)                       (read-out)
 *   and finally ht[n,h] = S^T.  Section "算子定位与算法背景" gives the update
 *   rule; section "算法原理" (M1-M4) gives the chunked evaluation with 128-token
 *   chunks that the library runs; section "算子签名与 I/O 规格" gives the
 *   tensors, dtypes and the [N, H, V, K] state layout; section "主机侧 wrapper
 *   与输入校验" gives fixed-length vs varlen packing and the rule that the
 *   host never reads cu_seqlens.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Calls are asynchronous on `stream`.  Argument checks happen on the host
 *     before anything is enqueued; a failed check enqueues nothing.
 *   - Errors are returned as kda_status; nothing is printed, nothing throws,
 *     the process is never terminated.  Faults the device detects (an invalid
 *     cu_seqlens, a wait that ran out) are recorded in the workspace status
 *     word and read with kda_get_status().
 *   - Tensor pointers must be 16-byte aligned (beta: 4-byte); the tensors are
 *     contiguous in the stated layout.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,     /* bad pointer, size, alignment or packing */
    KDA_ERR_UNSUPPORTED = 2,     /* K != 128 or V != 128 */
    KDA_ERR_CUDA = 3,            /* a CUDA runtime call failed */
    KDA_ERR_BAD_CU_SEQLENS = 4,  /* device found cu_seqlens invalid (via kda_get_status) */
    KDA_ERR_TIMEOUT = 5,         /* a bounded device wait ran out (via kda_get_status) */
    KDA_ERR_TOO_LARGE = 6,       /* kda_fwd_noalloc: the problem needs more workspace than
                                    the library's static scratch holds */
    KDA_ERR_BAD_STATE_INDEX = 7  /* kda_fused_recurrent: device found a state slot index or an
                                    accepted-token count out of range (via kda_get_status) */
} kda_status;

/* Apply the per-token L2 normalisation x / sqrt(sum(x^2) + 1e-6) to q and k
 * inside the kernel, before the scale (section "测试与验证体系" of the page). */
#define KDA_FLAG_QK_L2NORM 1u

/* kda_bwd only: run the token-by-token backward for every (sequence, head)
 * instead of the chunked one (fp32 throughout; slower). */
#define KDA_FLAG_BWD_TOKEN_EXACT 2u

/* kda_bwd only: evaluate every chunk's chain rule token by token in fp32 on
 * the CUDA cores instead of in chunked form on the tensor cores. */
#define KDA_FLAG_BWD_CHUNK_FP32 4u

/* kda_fwd only (training): also store the fp32 state entering every chunk, so
 * that a following kda_bwd on the same workspace with KDA_FLAG_BWD_REUSE_FWD
 * can skip its forward replay.  Needs a workspace of at least
 * kda_bwd_workspace_bytes(...) bytes; costs one extra write of the chunk
 * states (64 KiB per 128 tokens and head). */
#define KDA_FLAG_SAVE_FOR_BWD 8u

/* kda_bwd only: the workspace holds what the last kda_fwd with
 * KDA_FLAG_SAVE_FOR_BWD left in it (its tiles, flags and chunk states) for the
 * very same inputs (q, k, v, g, beta, scale, h0, cu_seqlens, sizes, q/k norm
 * flag), unchanged since: the backward skips its own forward replay.  The
 * caller guarantees that; nothing is checked.  Not with
 * KDA_FLAG_BWD_TOKEN_EXACT. */
#define KDA_FLAG_BWD_REUSE_FWD 16u

/* kda_fwd only: compute every (sequence, head) token by token with an fp32
 * state (the recurrence itself, the exact kernel the chunked path already
 * uses for units beyond its factoring range) instead of in chunked form.
 * For heads whose gates decay so slowly that the chunked path's fp16 product
 * operands exceed the final-state tolerance (about g/1000 per token and
 * slower); one sequential chain per (sequence, head, 32 value rows), so it
 * is much slower on long sequences.  Not with KDA_FLAG_SAVE_FOR_BWD. */
#define KDA_FLAG_FWD_TOKEN_EXACT 64u

/* kda_bwd only: evaluate the per-chunk chain rule with tcgen05 kind::tf32
 * products (operands staged K-major in shared memory, accumulators in TMEM)
 * instead of the default warp-level TF32 products.  Same results within the
 * backward's tolerance; slower on GB300 (its operand staging and transposes
 * are serialised with the products), kept as an alternative. */
#define KDA_FLAG_BWD_UMMA 32u

/*
 * Bytes of device workspace kda_fwd needs for these sizes (an upper bound
 * that covers both fixed-length and varlen packing).  0 on invalid sizes.
 * Layout: a 256-byte header (word 0 the device status; word 1 the number
 * of chunks the fast prep kernel queued for the wide one), the queue (one
 * int32 work item, slot * H + head, per queued chunk; room for every (chunk
 * slot, head), padded to 256 bytes), one 131584-byte tile per (128-token
 * chunk slot, head), then one flag word per (sequence, head).
 */
size_t kda_fwd_workspace_bytes(int B, int T, int H, int K, int V, int N);

/*
 * Chunked KDA forward.
 *
 *   q, k        bf16 [B, T, H, K]   queries / keys (row-major, contiguous)
 *   v           bf16 [B, T, H, V]
 *   g           fp32 [B, T, H, K]   log-domain forget gate, expected <= 0
 *   beta        fp32 [B, T, H]      delta-rule write strength
 *   scale       multiplier for q; <= 0 or NaN means K^-0.5
 *   h0          fp32 [N, H, V, K] initial state (transposed), or NULL for zero
 *   cu_seqlens  int32 [N+1] device offsets of N packed sequences (varlen,
 *               requires B == 1, cu[0] == 0, non-decreasing, cu[N] == T), or
 *               NULL for fixed length (N == B sequences of T tokens,
 *               T % 128 == 0).  Never read by the host.
 *   o           bf16 [B, T, H, V]   output (written for every valid token)
 *   ht          fp32 [N, H, V, K] final state, or NULL to skip it
 *   B, T, H, K, V, N  sizes (K == V == 128)
 *   flags       0 or KDA_FLAG_QK_L2NORM, with KDA_FLAG_SAVE_FOR_BWD or
 *               KDA_FLAG_FWD_TOKEN_EXACT
 *   workspace   device scratch of at least kda_fwd_workspace_bytes(...)
 *               bytes, 256-byte aligned; its contents need not be
 *               initialised.  Two calls that share a workspace must not
 *               overlap in time.
 *   stream      CUDA stream for every launch
 *
 * Precision: bf16 inputs, fp32 gate prefix sums, fp32 (I+A)^-1 and fp32
 * state; tensor-core products take fp16 operands with fp32 accumulation
 * (bf16 operands for the gated q.k / k.k products of chunks whose in-chunk
 * decay is too strong for fp16 factors).  v, and u = (I+A)^-1 diag(beta) v,
 * enter those products as fp16 in every chunk: they must stay below 65504
 * (fp16's largest value) in magnitude.
 * The gated products are factored around the chunk's middle row with
 * factors capped at e^80, exact (up to rounding) while the gate decay between
 * that row and the chunk's first or last row stays below 80 in each
 * dimension.  A (sequence, head) containing a chunk beyond that range is
 * recomputed exactly after the scan by the token-by-token recurrence (same
 * precision as kda_fused_recurrent), at token-by-token speed.
 */
kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht, int B,
                   int T, int H, int K, int V, int N, unsigned flags, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_fwd, additionally recording three caller-created CUDA events on
 * `stream`: stage_events[0] before the chunk-parallel kernel, [1] between it
 * and the sequential scan kernel, [2] after the scan.  Elapsed times between
 * them give each stage's device time inside a running sequence of calls.
 * Same arguments, contract and errors as kda_fwd; INVALID_ARG if any event
 * is null.
 */
kda_status kda_fwd_timed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht, int B,
                         int T, int H, int K, int V, int N, unsigned flags, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream, cudaEvent_t* stage_events);

/*
 * Synchronise `stream`, then read the device status word that the last
 * kda_fwd, kda_bwd or kda_fused_recurrent on this workspace wrote.  Returns KDA_OK,
 * KDA_ERR_BAD_CU_SEQLENS, KDA_ERR_TIMEOUT, KDA_ERR_BAD_STATE_INDEX (in that
 * order of precedence), or KDA_ERR_CUDA if synchronising or reading failed.
 */
kda_status kda_get_status(const void* workspace, cudaStream_t stream);

/*
 * Size of the static device scratch array behind kda_fwd_noalloc (64 MiB).
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * kda_fwd for callers that cannot allocate device memory: code running
 * inside a custom allocator's own callback (allocating there would re-enter
 * the allocator), a plug-in whose host application owns every allocation, or
 * a runtime with a fixed device-memory budget decided up front.  No
 * counterpart on the method's pages: it is a deployment convenience of this
 * library.
 *
 * Same arguments, layouts and precision as kda_fwd, minus the workspace: the
 * library uses a static __device__ array of KDA_NOALLOC_SCRATCH_BYTES that
 * every GPU which loads the library holds until the process exits.  Problems
 * with kda_fwd_workspace_bytes(...) > KDA_NOALLOC_SCRATCH_BYTES return
 * KDA_ERR_TOO_LARGE and enqueue nothing (at B=1 and H=8 that is T above about
 * 7,800 tokens).  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * The first call on each device looks up the array's device address with
 * cudaGetSymbolAddress (with that device current).  Every call on a device
 * shares the one array: calls whose GPU work overlaps in time (on different
 * streams, or from different host threads) race on it and give undefined
 * results, so serialise them.  kda_get_status() is not available for this entry point
 * (the status word lives in the shared array).
 */
kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                           float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht,
                           int B, int T, int H, int K, int V, int N, unsigned flags, cudaStream_t stream);

/*
 * Bytes of device workspace kda_fused_recurrent needs: the status word only.
 */
#define KDA_RECURRENT_WORKSPACE_BYTES 256u

/*
 * Token-by-token KDA with an in-place state pool: the decode-phase sibling
 * of kda_fwd (page "PyPTO-Gym chunk_kda operator", section "与其他 KDA 算子
 * 的关系": fused_recurrent_kda keeps an fp32 [H, V, K] state per sequence,
 * updates it in place at slots given by ssm_state_indices, supports
 * speculative decoding through num_accepted_tokens and the in-kernel q/k L2
 * normalisation).  Per token the same recurrence as kda_fwd (decay, delta
 * update, read-out), evaluated directly, one token after another.
 *
 *   q, k, v, g, beta, scale, cu_seqlens, o, B, T, H, K, V, N, flags
 *               as for kda_fwd, except that fixed-length T need not be a
 *               multiple of 128 (decode is typically T = 1 per sequence)
 *   state_pool  fp32 [pool_slots, H, V, K]: the states, read and written in
 *               place (same transposed layout as h0 / ht of kda_fwd)
 *   ssm_state_indices  int32 [N, indices_stride], device.  Row n names the
 *               slots of sequence n.
 *   num_accepted_tokens  int32 [N] device, or NULL.
 *     NULL (plain decode): sequence n starts from slot idx[n][0] and its
 *       final state is written back to that slot.  A negative slot marks a
 *       padding entry: the sequence is skipped, its output rows are zero
 *       and no state is read or written.
 *     non-NULL (speculative decoding): sequence n (at most indices_stride
 *       tokens) starts from slot idx[n][num_accepted_tokens[n] - 1], and the
 *       state after its token t is written to slot idx[n][t] (skipped where
 *       that slot is negative), so a verifier can resume from any accepted
 *       prefix.  num_accepted_tokens[n] must lie in [1, indices_stride].
 *     The pages name these two arguments without defining them further;
 *     this is the reading the library implements.
 *   workspace   device scratch of KDA_RECURRENT_WORKSPACE_BYTES, 256-byte
 *               aligned: the device status word, read with kda_get_status().
 *
 * Slots of different sequences must be distinct (two sequences writing one
 * slot race).  A slot >= pool_slots or an accepted count out of range sets
 * KDA_ERR_BAD_STATE_INDEX in the status word; that sequence's output rows
 * are zero and its states are left untouched.  An invalid cu_seqlens sets
 * KDA_ERR_BAD_CU_SEQLENS and the kernel does nothing for the bad entries.
 * Precision: fp32 state and arithmetic, bf16 output (round to nearest even).
 */
kda_status kda_fused_recurrent(const void* q, const void* k, const void* v, const float* g,
                               const float* beta, float scale, float* state_pool, int pool_slots,
                               const int32_t* ssm_state_indices, int indices_stride,
                               const int32_t* num_accepted_tokens, const int32_t* cu_seqlens, void* o,
                               int B, int T, int H, int K, int V, int N, unsigned flags, void* workspace,
                               cudaStream_t stream);

/*
 * Bytes of device workspace kda_kcp_fwd needs (0 on invalid sizes).
 */
size_t kda_kcp_workspace_bytes(int T, int H, int K, int V, int N, int world_size);

/*
 * Kimi Context Parallel (KCP) forward, with world_size ranks simulated on
 * this one device (page "flash-linear-attention KCP precision-debugging
 * guide": the single-device KCP simulator that loops over ranks and calls
 * the kernels directly).  The packed tokens [0, T) are cut into world_size
 * contiguous rank slices, rank r owning [T r / W, T (r+1) / W), which may
 * cut sequences anywhere.  Per rank: a pre-process computes, for its last
 * local piece, the transition M_r and the zero-start state S_ext,r (two
 * chunked forwards over that piece: v = 0 from the identity, and v from
 * zero); a merge in rank order gives the state entering each rank
 * (M_r S_start + S_ext,r); the local chunked forward then runs with that
 * state as the initial state of the rank's first piece.  The result equals
 * kda_fwd on the whole packed input up to rounding (chunk boundaries differ
 * where the rank cuts are not multiples of 128 inside a sequence, so
 * compare per token).
 *
 *   q, k, v, g, beta, scale, h0, o, ht, T, H, K, V, N, flags
 *               as for kda_fwd in varlen packing (B = 1)
 *   cu_seqlens_host  int32 [N+1] offsets in HOST memory: the rank split
 *               needs them on the host (validated there: BAD_CU_SEQLENS)
 *   world_size  number of simulated ranks, 1 .. 4096
 *   workspace   device scratch of kda_kcp_workspace_bytes(...) bytes,
 *               256-byte aligned
 *
 * The call synchronises `stream` once (after uploading the ranks' local
 * offsets) and is otherwise asynchronous.  kda_get_status(workspace)
 * reports the device status of the last internal forward.
 */
kda_status kda_kcp_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                       const float* h0, const int32_t* cu_seqlens_host, void* o, float* ht, int T, int H, int K,
                       int V, int N, int world_size, unsigned flags, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/*
 * Number of CTAs (and of 8 MiB per-CTA scratch buffers) the token-by-token
 * backward runs at most.
 */
#define KDA_BWD_EXACT_MAX_CTAS 152

/*
 * Bytes of device workspace kda_bwd needs for these sizes (0 on invalid
 * sizes).  Layout: the kda_fwd workspace (status header, forward tiles,
 * flags), a second tile per (128-token chunk slot, head) for the reverse
 * state pass, three fp32 K x V states per (chunk slot, head) (chunk states,
 * state gradients, and the token-by-token path's chunk states), one word
 * per (chunk slot, head) marking chunks left to the per-token kernel, then
 * min(max(chunk slots x H, N x H), KDA_BWD_EXACT_MAX_CTAS) scratch buffers of
 * 128 states.
 */
size_t kda_bwd_workspace_bytes(int B, int T, int H, int K, int V, int N);

/*
 * KDA backward: the gradients of L = sum_t <dout_t, o_t> + sum_n <dht_n, ht_n>
 * with respect to q, k, v, g, beta and h0, where (o, ht) is the kda_fwd
 * forward of the same arguments.  The page lists the backward kernels of the
 * training path (dv, dq/dk/dw/dg, the state gradient dh and the WY
 * back-propagation) but gives no formulas; this entry point computes their
 * plain definition, the vector-Jacobian product of the per-token recurrence
 * documented at the top of this file.
 *   q, k, v, g, beta, scale, h0, cu_seqlens, B, T, H, K, V, N, flags
 *               as for kda_fwd (the same forward is differentiated)
 *   dout        bf16 [B, T, H, V]   dL/do
 *   dht         fp32 [N, H, V, K]   dL/dht, or NULL for zero
 *   dq, dk      fp32 [B, T, H, K]   written for every valid token (with
 *               KDA_FLAG_QK_L2NORM: gradients with respect to the raw,
 *               unnormalised q and k)
 *   dv          fp32 [B, T, H, V]
 *   dg          fp32 [B, T, H, K]
 *   dbeta       fp32 [B, T, H]
 *   dh0         fp32 [N, H, V, K]   dL/dh0 (also when h0 is NULL: the
 *               gradient at the zero state), or NULL to skip it
 *   workspace   device scratch of at least kda_bwd_workspace_bytes(...)
 *               bytes, 256-byte aligned, contents need not be initialised;
 *               calls sharing it must not overlap in time
 * Method (chunked path, the default): the forward's chunk-parallel kernel
 * and its scan (state only) give the fp32 state entering every 128-token
 * chunk; the state gradient obeys the same recurrence with the transposed
 * transition, dS_c = Dg_c dS_{c+1} + Nm_c^T dS_{c+1} + Qe_c^T do_c, which the
 * same scan evaluates on transposed tiles in reverse chunk order; then every
 * chunk applies the chain rule in chunked form from its entering state and
 * its exit state gradient, on TF32 tensor-core products (with
 * KDA_FLAG_BWD_CHUNK_FP32: token by token in fp32; chunks outside the
 * chunked form's factor range take that path anyway).  Precision: the chunk
 * states and state gradients carry the forward's product precision (fp16
 * operands, fp32 accumulation), the per-chunk part TF32 products with fp32
 * accumulation.  Range: the reverse pass takes Qe_c^T do_c as fp16, so its
 * entries must stay below 65504 and lose relative precision below about
 * 6e-5 (fp16's normal range); dout of the magnitudes loss scaling produces
 * keeps them inside it.
 * (sequence, head) units the forward flags as beyond its factoring range go
 * to the token-by-token path, which replays the forward in fp32 one token at
 * a time (exact for any decay, one unit per CTA: slow); with
 * KDA_FLAG_BWD_TOKEN_EXACT every unit takes it.
 * Errors: as for kda_fwd; an invalid cu_seqlens is reported through
 * kda_get_status(workspace).
 */
kda_status kda_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                   const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq,
                   float* dk, float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K, int V,
                   int N, unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_bwd (chunked path), additionally recording six caller-created CUDA
 * events on `stream`: [0] at the start, [1] after the forward replay (the
 * chunk-parallel kernel and the state pass that stores the chunk states),
 * [2] after the transposed tiles, [3] after the reverse state pass, [4] after
 * the per-chunk chain-rule kernel, [5] at the end (after the token-by-token
 * kernel for flagged units and the normalisation chain rule).  Same
 * arguments and contract as kda_bwd; INVALID_ARG if any event is null or
 * KDA_FLAG_BWD_TOKEN_EXACT is set.
 */
kda_status kda_bwd_timed(const void* q, const void* k, const void* v, const float* g, const float* beta, float scale,
                         const float* h0, const int32_t* cu_seqlens, const void* dout, const float* dht, float* dq,
                         float* dk, float* dv, float* dg, float* dbeta, float* dh0, int B, int T, int H, int K, int V,
                         int N, unsigned flags, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         cudaEvent_t* stage_events);

/* Static English description of a status code. */
const char* kda_status_str(kda_status status);

/*
 * Test hooks for the failure detection of the bounded device waits (no
 * counterpart on the pages; the pages' kernels have no such waits).  Every
 * wait of one CTA role on another (tensor-core product done, bulk copy
 * landed, a stage freed) polls at most a fixed number of times; when one
 * runs out the CTA records KDA_ERR_TIMEOUT in the workspace status word,
 * every later wait of that CTA returns at once, the CTA waits for the copies
 * and products it issued itself, frees its tensor memory and exits.
 *   KDA_DEBUG_WAIT_LIMIT: poll limit of those waits for the following calls
 *     (value 0 restores the default, 2^24 polls).
 *   KDA_DEBUG_DROP_SCAN_LOAD: the next kda_fwd only (the hook resets itself
 *     when that call is enqueued): in the sequential scan, unit (sequence 0,
 *     head 0), value tile 0 never issues the load of chunk 1's stage, so the
 *     waits on it run out.  Needs a sequence of at least two chunks.
 * The settings are process-wide and not synchronised: set them only while no
 * other thread calls the library.  Returns KDA_ERR_INVALID_ARG for an
 * unknown `what`.
 */
#define KDA_DEBUG_WAIT_LIMIT 1
#define KDA_DEBUG_DROP_SCAN_LOAD 2
kda_status kda_debug_set(int what, unsigned value);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
