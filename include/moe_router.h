/*
 * moe_router.h -- C ABI of the GB300 (sm_103a) MoE expert-routing library.
 *
 * The hot path of MoE expert routing with equal-cost load balancing: router
 * softmax and top-k, the Switch auxiliary balance loss and its closed-form
 * gradient, a capacity-limited stable token->expert dispatch, and the batched
 * topology-aware Sinkhorn-Knopp flow plan of TAOT Phase 1.  Beside them: the
 * aux-loss-free bias routing, the masked P_i variant and the full router
 * backward through the gates, the batch statistics of data-parallel shards,
 * the EPLB replication / packing planner, and TAOT Phase 2 (column-first
 * matching of hot experts to cold ranks).
 *
 * Sources (cited by title and section):
 *   [P1] the three-layer load-balancing article (LVS, NIC Teaming, MoE
 *        equal-cost balancing), mhpq.cn/news/998159
 *   [P2] "MoE大模型训练中的等开销负载均衡：原理、代码实现与调参实战" (codechina.net)
 *   [P3] large-model load-balancing survey printed as "企业官网建设流程全解析"
 *        (cnvsn.com/news/335486)
 *   [P4] "MoE 训练端到端加速 1.43 倍：LoongForge 基于拓扑感知最优传输重新定义 EP
 *        专家负载均衡" (LoongForge blog, TAOT)
 *
 * Conventions for every entry point:
 *   - Array arguments are DEVICE pointers owned by the caller, dense and
 *     row-major, unless a comment says otherwise.  The library never
 *     allocates device memory; scratch lives in a caller-allocated workspace.
 *   - Work is enqueued on `stream` (0 = the legacy default stream) and the
 *     call returns without synchronising.  Results are valid once the stream
 *     reaches that point.  Calls that share a workspace must be ordered on one
 *     stream; concurrent calls need separate workspaces.
 *   - The persistent kernels (moe_router_fwd, moe_dispatch, moe_router_step)
 *     are launched with programmatic dependent launch: a launch may be
 *     scheduled while the previous kernel of the stream finishes and waits
 *     for it before touching memory, and each launch lets the next one be
 *     scheduled once all its CTAs have passed their grid barrier.  A kernel
 *     of the caller's that is itself launched with programmatic stream
 *     serialization must wait for its prerequisite grid
 *     (cudaGridDependencySynchronize) before it reads these outputs; any
 *     other launch is ordered as usual.
 *   - Errors are returned as moe_status; no exception crosses the ABI.
 *     Argument errors are found on the host before anything is enqueued.
 *     moe_last_error() gives a one-line description of the last failure on
 *     the calling thread.
 *   - Inputs are assumed finite: NaN or Inf logits give unspecified results.
 *   - Indices are int32; T*k must stay below 2^31.
 */
#ifndef MOE_ROUTER_H
#define MOE_ROUTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Version of this interface (moe_abi_version returns it).
 *   1: the router step, its parts, the Sinkhorn plan, bias routing, the full
 *      backward, EPLB, TAOT Phase 2 and the shard combine;
 *   2: adds moe_router_step_ex (the bias-routed step in one launch),
 *      moe_shard_capacity_base and moe_dispatch_sharded (the capacity of a
 *      batch split over data-parallel ranks).  Version 1 calls are unchanged. */
#define MOE_ROUTER_ABI_VERSION 2

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,     /* bad argument: null pointer, size out of range, misaligned workspace */
  MOE_ERR_UNSUPPORTED = 2, /* unknown dtype */
  MOE_ERR_CUDA = 3,        /* a CUDA launch or query failed (moe_last_error has the CUDA message) */
  MOE_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (see moe_get_device_status) */
  MOE_ERR_WORKSPACE = 5    /* workspace smaller than the *_workspace_size query asked for */
} moe_status;

typedef enum { MOE_DTYPE_FP32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

/* Indices into the `scalars` output of moe_router_fwd / moe_router_step. */
enum {
  MOE_SCALAR_L_AUX = 0,              /* alpha * E * sum_i f_i P_i                        */
  MOE_SCALAR_BALANCE = 1,            /* E * sum_i f_i P_i (1 under uniform routing)      */
  MOE_SCALAR_CV = 2,                 /* std/mean of the per-expert counts (population)   */
  MOE_SCALAR_MAX_OVER_MEAN = 3,      /* max count / mean count                           */
  MOE_SCALAR_MIN_OVER_MEAN = 4,      /* min count / mean count                           */
  MOE_SCALAR_RANK_CV = 5,            /* std/mean of the per-rank loads (0 if n_ranks==0) */
  MOE_SCALAR_RANK_MAX_OVER_MEAN = 6, /* max rank load / mean rank load (0 if none)       */
  MOE_NUM_SCALARS = 7
};

/* Limits checked by every entry point (MOE_ERR_INVALID otherwise). */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 8
#define MOE_MAX_RANKS 64

/* ------------------------------------------------------------------------ */
/* Workspace                                                                */
/* ------------------------------------------------------------------------ */

/* Bytes of device scratch that moe_router_fwd, moe_dispatch and
 * moe_router_step need for a batch of T tokens over E experts with top-k.
 * Returns 0 for arguments that those calls would reject. */
MOE_API size_t moe_router_workspace_size(int64_t T, int32_t E, int32_t k);

/* Zero-fills a workspace (an async memset on `stream`).  A workspace must be
 * zero-filled once before its first use; every call that completes leaves it
 * ready for the next one.  After a call reported MOE_ERR_TIMEOUT, initialise
 * it again.  `ws` must be 256-byte aligned. */
MOE_API moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Reads and clears the device error flags of a workspace (synchronises
 * `stream`).  *flags = 0 when every bounded wait completed; otherwise
 * returns MOE_ERR_TIMEOUT and sets bits: 1 = grid barrier wait expired,
 * 2 = a wait of the kernel's internal pipeline expired.  With ws = NULL it
 * reads and clears the flags of moe_router_step_static's fixed scratch on
 * the current device instead. */
MOE_API moe_status moe_get_device_status(void* ws, moe_stream_t stream, int32_t* flags);

/* ------------------------------------------------------------------------ */
/* Router forward                                                           */
/* ------------------------------------------------------------------------ */

/* Router softmax, top-k and the Switch balance statistics of one batch.
 *
 * Computes, in fp32 from fp32 or bf16 logits:
 *   p[t,e]  = softmax(logits[t,:])[e]                        [P1] §4.2; [P2] §3.1
 *   idx[t,j]: the k experts with the largest logits, largest first, ties to
 *             the lower expert index                        [P1] §4.4; [P2] §3.1
 *   gate[t,j] = p[t, idx[t,j]], divided by sum_j p[t, idx[t,j]] when renorm
 *   counts[e] = #assignments to e (before capacity drops)    [P2] §3.1 (bincount, minlength=E)
 *   f[e]      = counts[e] / (T*k)                            [P1] §4.4
 *   P[e]      = (1/T) * sum_t p[t,e]  (all tokens, unmasked) [P1] §4.2
 *   scalars   = MOE_SCALAR_*: L_aux = alpha*E*sum f*P ([P2] §2.2), the
 *               balance E*sum f*P, CV and max/min over mean of the counts
 *               ([P3] §5.1), and the same over ranks
 *   rank_load[r] = sum of counts over experts [r*E/n_ranks, (r+1)*E/n_ranks)
 *
 * logits     [T,E] fp32 or bf16 (dt).
 * k          1..min(E, 8).     E in 1..1024.     T >= 1, T*k < 2^31.
 * alpha      >= 0, the aux-loss weight applied inside L_aux.
 * renorm     1: renormalise the gate over the picks; 0: raw p; -1: auto (k > 1).
 * n_ranks    0 for none, else 1..64 dividing E (experts mapped contiguously).
 * idx [T,k] int32, gate [T,k] fp32, counts [E] int32, f [E] fp32, P [E] fp32,
 * scalars [MOE_NUM_SCALARS] fp32, rank_load [n_ranks] int32 (may be NULL
 * when n_ranks == 0).  ws: >= moe_router_workspace_size(T,E,k) bytes,
 * 256-byte aligned, zero-filled before first use.
 * The per-expert results are reduced in a fixed order: repeated calls give
 * bit-identical outputs. */
MOE_API moe_status moe_router_fwd(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                          float alpha, int32_t renorm, int32_t n_ranks,
                          int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                          float* scalars, int32_t* rank_load,
                          void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Router backward (aux loss only)                                          */
/* ------------------------------------------------------------------------ */

/* Gradient of grad_scale * L_aux with respect to the logits, f held constant
 * (f comes from the hard top-k selection and carries no gradient, [P1] §4.2):
 *
 *   dlogits[t,j] = grad_scale * (alpha*E/T) * p[t,j] * (f[j] - sum_i p[t,i] f[i])
 *
 * logits [T,E] fp32/bf16, f [E] fp32 (as written by moe_router_fwd),
 * dlogits [T,E] fp32 (written, not accumulated).  No workspace. */
MOE_API moe_status moe_router_bwd(const void* logits, moe_dtype dt, int64_t T, int32_t E, float alpha,
                          const float* f, float grad_scale, float* dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Capacity-limited dispatch                                                */
/* ------------------------------------------------------------------------ */

/* Expert capacity C = ceil(ceil(T*k/E) * capacity_factor), the product in
 * double ([P1] §4.5: 1024 tokens, 8 experts, factor 1.25 -> 160).  Host-only.
 * Returns -1 for invalid arguments (T < 1, E < 1, k < 1, factor <= 0). */
MOE_API int64_t moe_dispatch_capacity(int64_t T, int32_t E, int32_t k, double capacity_factor);

/* Stable counting-sort dispatch of the T*k assignments a = t*k + j by expert
 * with capacity C = moe_dispatch_capacity(T,E,k,capacity_factor) ([P1] §4.5:
 * assignments beyond an expert's capacity are dropped):
 *   offsets [E+1] int32: exclusive prefix of the per-expert counts, offsets[E] = T*k
 *   perm    [T*k] int32: assignment ids grouped by expert, ascending within an expert
 *   slot    [T*k] int32: rank of assignment a within its expert, -1 if >= C (dropped)
 *   kept    [E]   int32: min(count, C)
 *   n_dropped [1] int32: T*k - sum(kept)
 * The kept assignments of expert e are perm[offsets[e] .. offsets[e]+kept[e]).
 * idx [T,k] int32 with values in [0,E) (out-of-range values give unspecified
 * results but stay in bounds).  capacity_out: HOST pointer, may be NULL.
 * ws as for moe_router_fwd. */
MOE_API moe_status moe_dispatch(const int32_t* idx, int64_t T, int32_t E, int32_t k, double capacity_factor,
                        int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                        int32_t* n_dropped, int64_t* capacity_out,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* Global capacity across data-parallel ranks.  The capacity of [P1] §4.5 is
 * that of the whole batch, and a batch split over G data-parallel ranks (rank
 * g holding the rows after those of ranks 0..g-1) is dispatched as if one
 * call had taken all of it: an assignment's position in its expert's buffer
 * counts the expert's assignments on the lower ranks first.
 *
 * moe_shard_capacity_base writes cap_base[e] = sum over ranks g < rank of
 * counts[g][e] (summed in 64 bits, clamped to INT32_MAX): the exclusive scan
 * across ranks of every expert's count.  counts [G,E] int32 device, the ranks'
 * per-expert counts stacked in rank order (on a multi-GPU job the result of an
 * all-gather of moe_router_fwd's counts); cap_base [E] int32 device.  G in
 * [1,64], rank in [0,G).  One small launch, no workspace. */
MOE_API moe_status moe_shard_capacity_base(const int32_t* counts, int32_t G, int32_t E, int32_t rank,
                                   int32_t* cap_base, moe_stream_t stream);

/* moe_dispatch of one rank's T rows of a batch of T_total rows, with the
 * batch's capacity C = moe_dispatch_capacity(T_total, E, k, capacity_factor)
 * and cap_base [E] (device) from moe_shard_capacity_base:
 *   perm, offsets: as moe_dispatch, over this rank's assignments (local ids)
 *   slot [T*k]:    cap_base[e] + r when that is below C, else -1, r the
 *                  assignment's rank among this rank's assignments to e
 *   kept [E]:      min(count_e, max(C - cap_base[e], 0)), count_e this rank's
 *   n_dropped [1]: T*k - sum(kept)
 * Over all ranks, the slots (concatenated in rank order) are moe_dispatch's
 * slots of the whole batch, the kept sum to its kept, the n_dropped to its
 * n_dropped.  Errors: T_total < T, T_total*k >= 2^31, cap_base NULL or not
 * 4-byte aligned, and everything moe_dispatch rejects.  ws as for
 * moe_router_fwd. */
MOE_API moe_status moe_dispatch_sharded(const int32_t* idx, int64_t T, int32_t E, int32_t k, double capacity_factor,
                                int64_t T_total, const int32_t* cap_base,
                                int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                int32_t* n_dropped, int64_t* capacity_out,
                                void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused step: forward + dispatch + backward in one launch                  */
/* ------------------------------------------------------------------------ */

/* One pass of the whole hot path over a batch: exactly the outputs of
 * moe_router_fwd, then moe_dispatch on the idx it produced, then
 * moe_router_bwd with its f, computed by one persistent cooperative kernel
 * (grid-wide barriers separate the global reductions).  Outputs are
 * bit-identical to the three separate calls, with one exception: for bf16
 * logits with 129 <= E <= 512 and renormalised gates the step forms the
 * rows' softmax sums and P in its backward, and P (with L_aux and the
 * balance, which use it) is then the exact sum of other partial sums, equal
 * to moe_router_fwd's to rounding (both within the stated tolerance of the
 * exact value) and bit-identical from run to run.  Arguments as above. */
MOE_API moe_status moe_router_step(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                           float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                           float grad_scale,
                           int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                           float* scalars, int32_t* rank_load,
                           int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                           int32_t* n_dropped, float* dlogits,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* The extended training step in one launch: the outputs of moe_router_fwd_ex
 * (bias routing with the bias update, masked P), then moe_dispatch on its idx,
 * then moe_router_bwd_full with its f and the given upstream gradient of the
 * gates, computed by one persistent cooperative kernel:
 *   - selection on s = fp32(z) + bias_e ([P1] §4.3: the bias moves the choice
 *     of experts only); softmax, gates and P from the unbiased z; bias NULL
 *     means zero bias;
 *   - masked_p != 0: P_i = (1/(T*k)) sum_t p[t,i] [i picked by t] ([P2] §3.1)
 *     in P, the balance and L_aux, and in the gradient of the aux loss;
 *   - bias_out != NULL: bias_out[e] = bias[e] + bias_gamma * sign(T*k/E -
 *     counts[e]) in fp32 (sign(0) = 0); bias_out may alias bias;
 *   - dlogits = dL/dlogits of L = sum_{t,j} dgate[t,j] * gate[t,j] +
 *     grad_scale * L_aux, the picks and f held fixed; dgate [T,k] fp32 may be
 *     NULL (the aux loss alone).
 * The other arguments, the outputs and the workspace are those of
 * moe_router_step.  idx, counts, perm, slot, offsets, kept, n_dropped and
 * bias_out are bit-identical to the three separate calls'; gate, f, P, the
 * scalars and dlogits agree within fp32 rounding (the separate forward sums p
 * in fixed point, this step in fp32 per CTA).  Errors: those of
 * moe_router_step, and INVALID for a bias, bias_out or dgate that is not
 * 4-byte aligned or a non-finite bias_gamma with bias_out given. */
MOE_API moe_status moe_router_step_ex(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                              float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                              float grad_scale, const float* bias, float bias_gamma, float* bias_out,
                              int32_t masked_p, const float* dgate,
                              int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                              float* scalars, int32_t* rank_load,
                              int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                              int32_t* n_dropped, float* dlogits,
                              void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_router_step for inputs and outputs in HOST memory.
 *
 * One call queues, on `stream`: the copy of the logits from host memory into
 * a caller-owned device staging buffer, moe_router_step on it, and the copy
 * of every output of the step (idx, gate, counts, f, P, scalars, rank_load,
 * perm, slot, offsets, kept, n_dropped, dlogits) back to the host arrays.
 * It is asynchronous: the host arrays hold the results once the stream has
 * reached the end of the call.  The host arrays should be page-locked
 * (cudaHostAlloc / cudaHostRegister); with pageable memory CUDA stages the
 * copies and the call blocks the host.
 *   - logits and every output pointer are HOST pointers with the layouts of
 *     moe_router_step (rank_load may be NULL when n_ranks == 0).
 *   - dev: a caller-owned device buffer of at least
 *     moe_router_step_host_device_size(dt, T, E, k, n_ranks) bytes, 256-byte
 *     aligned (MOE_ERR_WORKSPACE if smaller).  It is overwritten.
 *   - ws, ws_bytes: the step's workspace, as for moe_router_step.
 *   - kernel_after, kernel_done: cudaEvent_t handles or NULL.  The step's
 *     kernel waits for kernel_after (cudaStreamWaitEvent, after the logits'
 *     copy has been queued) and kernel_done is recorded right after it, so
 *     that calls alternating between streams can overlap one call's copies
 *     with another's kernel while the kernels themselves run one at a time.
 *   - Calls that overlap in time (several streams) need their own dev and ws.
 * Errors: those of moe_router_step, MOE_ERR_INVALID for a NULL host pointer,
 * MOE_ERR_CUDA when a copy cannot be queued. */
MOE_API size_t moe_router_step_host_device_size(moe_dtype dt, int64_t T, int32_t E, int32_t k, int32_t n_ranks);
MOE_API moe_status moe_router_step_host(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                                        float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                                        float grad_scale,
                                        int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                                        float* scalars, int32_t* rank_load,
                                        int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                        int32_t* n_dropped, float* dlogits,
                                        void* dev, size_t dev_bytes, void* ws, size_t ws_bytes,
                                        void* kernel_after, void* kernel_done, moe_stream_t stream);

/* moe_router_step for callers that cannot allocate device memory.
 *
 * Not a step of the method: the source pages have no counterpart.  It exists
 * for callers that can pass inputs and outputs but cannot allocate or lend
 * scratch memory: code running where allocation is not allowed or not safe,
 * plugins with a device-memory budget fixed at load time, or runtimes that
 * keep all device memory in their own pool.  Its scratch is a fixed array
 * inside the library image (4.75 MiB, held by every GPU that loads the
 * library until the process exits); the call allocates nothing and frees
 * nothing.
 *   - Arguments and outputs are exactly those of moe_router_step, minus the
 *     workspace; the results are the same, bit for bit.
 *   - E must be <= 512 (MOE_ERR_INVALID otherwise, with a message naming the
 *     limit).  Every argument is checked before anything is queued, so a
 *     refused call leaves the shared array untouched.
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress, with that device current) and caches it for the
 *     life of the process; make that first call before any stream capture.
 *     The cache assumes the device's primary context is never reset: after a
 *     cudaDeviceReset the library's module, and the array with it, may be
 *     loaded at another address, so do not call this entry point again in
 *     that process.
 *   - All calls on a device share the one array: calls that may overlap on the
 *     GPU (different streams, or different host threads) race.  Each call
 *     clears the array's barrier count, counters and group sums on `stream`
 *     before its kernel.
 *   - An expired device wait (MOE_ERR_TIMEOUT in moe_router_step's terms)
 *     leaves its error bits set in the array; later calls then write nothing
 *     until moe_get_device_status(NULL, stream, &flags) reads the bits,
 *     returns MOE_ERR_TIMEOUT and clears them. */
MOE_API moe_status moe_router_step_static(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                                          float alpha, int32_t renorm, int32_t n_ranks, double capacity_factor,
                                          float grad_scale,
                                          int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                                          float* scalars, int32_t* rank_load,
                                          int32_t* perm, int32_t* slot, int32_t* offsets, int32_t* kept,
                                          int32_t* n_dropped, float* dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Aux-loss-free bias routing, masked P_i, full backward through the gates   */
/* ------------------------------------------------------------------------ */

/* Router forward with two options of the method that moe_router_fwd does not
 * take, computed by the persistent cooperative kernel of moe_router_fwd (the
 * forward phases of moe_router_step_ex; per-expert sums added in a fixed
 * order, so repeated calls give the same bits):
 *
 *   Bias routing ([P1] §4.3, aux-loss-free balancing): each expert carries a
 *   scalar bias b_e on its router logit that steers which experts are picked.
 *   Top-k ranks s[t,e] = fp32(z[t,e]) + b_e (one fp32 addition, round to
 *   nearest; ties to the lower expert index); softmax, gates, P and the
 *   backward use the unbiased z.  bias [E] fp32, or NULL for b = 0.
 *   With bias_out non-NULL the call also writes the updated bias
 *       bias_out[e] = b_e + bias_gamma * sign(T*k/E - counts[e])
 *   (the sign from the exact integer comparison of counts[e]*E with T*k,
 *   sign 0 -> no change; one fp32 addition): an overloaded expert's bias goes
 *   down, an idle one's up.  bias_out may alias bias (in-place update).
 *
 *   Masked P ([P2] §3.1, the code of [P1] §4.4): with masked_p != 0,
 *       P[e] = (1/(T*k)) * sum_t p[t,e] * [e is one of t's picks]
 *   instead of the unmasked mean (1/T) sum_t p[t,e] ([P1] §4.2).  balance and
 *   L_aux use this P.
 *
 * Every other argument and output is that of moe_router_fwd (same layout,
 * same scalars, same workspace size: moe_router_workspace_size; the
 * workspace must have been zeroed once by moe_workspace_init and is left
 * reusable).  With bias = NULL and masked_p = 0 the picks and counts equal
 * moe_router_fwd's bit for bit, the floating outputs to rounding.
 * bias_gamma must be finite.  Its one grid barrier waits with the bounded
 * wait of moe_router_fwd (an expired wait: moe_get_device_status). */
MOE_API moe_status moe_router_fwd_ex(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                             float alpha, int32_t renorm, int32_t n_ranks,
                             const float* bias, int32_t masked_p, float bias_gamma, float* bias_out,
                             int32_t* idx, float* gate, int32_t* counts, float* f, float* P,
                             float* scalars, int32_t* rank_load,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* Full router backward: the gradient with respect to the logits of
 *     L = sum_{t,j} dgate[t,j] * gate[t,j](z)  +  grad_scale * L_aux(z),
 * the picks idx and f held constant (top-k is piecewise constant; f carries
 * no gradient, [P1] §4.2).  dgate [T,k] fp32 is the main loss's upstream
 * gradient of the gates written by the forward; gate[t,j] = p[t,idx[t,j]]
 * (renorm = 0) or that p divided by the sum of the row's picked p (renorm = 1;
 * -1 = automatic: renorm iff k > 1).  L_aux uses the unmasked P_i, or the
 * masked P_i with masked_p != 0 (then its gradient reaches the picked logits
 * only through P).  Per row, with dp the gradient with respect to p:
 *     dlogits[t,j] = p[t,j] * (dp[t,j] - sum_i p[t,i] dp[t,i]).
 * dgate may be NULL (aux loss only: with masked_p = 0 this is moe_router_bwd);
 * idx [T,k] int32 is required when dgate is given or masked_p != 0, else may
 * be NULL; its values must lie in [0,E) (others give unspecified results but
 * every access stays in bounds).  dlogits [T,E] fp32 is written, not
 * accumulated.  No workspace. */
MOE_API moe_status moe_router_bwd_full(const void* logits, moe_dtype dt, int64_t T, int32_t E, int32_t k,
                               float alpha, const float* f, float grad_scale, int32_t masked_p,
                               const int32_t* idx, const float* dgate, int32_t renorm,
                               float* dlogits, moe_stream_t stream);

/* Data-parallel batch statistics.  Combines the forward statistics of G shards
 * of one batch -- data-parallel ranks that each routed their own tokens with
 * moe_router_fwd / moe_router_fwd_ex, or slices routed one after another --
 * into the whole batch's, as if one call had routed all of it:
 *   counts = sum_s counts_s (exact),  P = sum_s P_s * T_s / T  (double, then fp32;
 *   the same for masked P),  f = counts / (T*k),  the scalars and rank loads as
 *   moe_router_fwd computes them, T = sum_s T_s.
 * counts [G,E] int32 and P [G,E] fp32 are the shards' outputs stacked (on a
 * multi-GPU job, the result of an all-gather); T_shard is a HOST array of G
 * token counts.  G in [1,64].  The batch gradient then comes from each shard's
 * moe_router_bwd with the combined f and grad_scale * T_s / T (its coefficient
 * alpha*E/T_s becomes alpha*E/T).  No workspace; one CTA. */
MOE_API moe_status moe_router_combine(const int32_t* counts, const float* P, const int64_t* T_shard, int32_t G,
                              int32_t E, int32_t k, float alpha, int32_t n_ranks, int32_t masked_p,
                              int32_t* counts_out, float* f, float* P_out, float* scalars, int32_t* rank_load,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* EPLB: expert replication and balanced packing onto GPUs                  */
/* ------------------------------------------------------------------------ */

/* [P3] §4.1.2, for B independent problems (layers or microbatches) at once,
 * one CTA each.  loads [B,E] int32: tokens routed to each expert (>= 0; the
 * counts moe_router_fwd writes).
 *   replicate_experts: starting from one copy per expert, repeatedly add a
 *     copy of the expert whose load per copy w/c is largest (compared
 *     exactly, w_a*c_b against w_b*c_a; ties to the lower index) until there
 *     are num_phys copies;
 *   balanced_packing: items heaviest first, each into the currently lightest
 *     bin that is not yet full, every bin taking the same number of items (in
 *     fp32: a copy weighs fp32(w)/fp32(c), a bin's total is the fp32 sum of
 *     its items in placement order; ties to the lower item / bin index).
 * Policy: hierarchical when num_groups > 0 and num_nodes divides num_groups
 * (experts form num_groups contiguous groups; groups are packed onto nodes by
 * their summed load, then each node's experts, in the order its groups were
 * placed, are replicated onto num_phys/num_nodes slots and packed onto its
 * num_gpus/num_nodes GPUs, node n owning GPUs [n*G/N, (n+1)*G/N)); global
 * otherwise (replication over all E experts, packing onto all GPUs).
 * Outputs:
 *   phy2log   [B,num_phys] int32: the logical expert in each physical slot;
 *             GPU g holds slots [g*S, (g+1)*S), S = num_phys/num_gpus, in the
 *             order the packing placed them
 *   log_count [B,E] int32: copies of each expert (sums to num_phys)
 *   gpu_load  [B,num_gpus] fp32: each GPU's load, the sum of w/c over its copies
 * Limits: E in [1,1024]; num_phys in [E, 4096], a multiple of num_gpus;
 * num_gpus in [1,256], a multiple of num_nodes >= 1; num_groups 0 or a
 * divisor of E.  No workspace. */
MOE_API moe_status moe_eplb_plan(const int32_t* loads, int32_t B, int32_t E, int32_t num_phys,
                         int32_t num_gpus, int32_t num_nodes, int32_t num_groups,
                         int32_t* phy2log, int32_t* log_count, float* gpu_load, moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* TAOT Phase 1: batched topology-aware Sinkhorn flow plan                  */
/* ------------------------------------------------------------------------ */

/* [P4] §2 Phase 1 and §3: per microbatch m, the overloaded ranks' excess load
 * is a supply and the idle ranks' spare capacity a demand:
 *   a_r = max(load_r - mean, 0) / sum,  b_r = max(mean - load_r, 0) / sum
 * The cost is W[r,s] = 0 (same rank), 1 (same node), lambda (across nodes),
 * rank r on node r / ranks_per_node; the Gibbs kernel M = exp(-W/eps).
 * Starting from v = 1, `iters` times: u = a / max(M v, 1e-30), then
 * v = b / max(M^T u, 1e-30).  The plan is diag(u) M diag(v).
 *
 * loads [B,R] fp32; R in 1..64; ranks_per_node in 1..R dividing R;
 * lambda > 0; eps <= 0 means eps = lambda; iters >= 0.
 * u, v [B,R] fp32; plan [B,R,R] fp32 or NULL; status [B] int32:
 * 0 = planned, 1 = nothing to move (no rank above the mean; u = v = plan = 0).
 * One warp per microbatch, O(R) work per iteration (M has three distinct
 * values, so M x needs only x, its per-node sums and its total); no workspace. */
MOE_API moe_status taot_sinkhorn_batched(const float* loads, int32_t B, int32_t R, int32_t ranks_per_node,
                                 float lambda, float eps, int32_t iters,
                                 float* u, float* v, float* plan, int32_t* status,
                                 moe_stream_t stream);

/* TAOT Phase 2 ([P4] §2, §3): column-first matching of hot experts to cold
 * ranks, for B microbatches at once (one CTA each).  Experts live on their home
 * ranks contiguously (E/R per rank); a rank is hot above the mean load, cold
 * below it.  Rounds repeat until no cold rank finds a match (at most R*K + 1):
 * every cold rank with a free slot (at most K replicas each) picks the hot expert
 * that scores best,
 *   (tokens moved x, 1 if same node else 0, plan[h,c], then the lower expert),
 *   x = min(tokens of e still at home, floor(load[h] - mean), floor(mean - load[c])),
 * skipping experts it already holds; several ranks picking one expert are
 * arbitrated by the same score (ties to the lower rank); the winners' moves are
 * applied in ascending rank order, each x taken again against the current
 * loads.  The page gives the three levels of the score and the arbitration,
 * not these formulas: they are this library's reading.
 * expert_loads [B,E] int32 (>= 0, total per microbatch below 2^31);
 * plan [B,R,R] fp32, the Phase 1 flow (taot_sinkhorn_batched's plan);
 * R in [1,64] dividing E; ranks_per_node dividing R; K in [0,16]; E <= 1024.
 * Outputs: slot_expert [B,R,K] int32 (the expert in cold rank r's j-th
 * replica slot, -1 when empty), slot_tokens [B,R,K] int32 (tokens it takes),
 * rank_load [B,R] int32 (loads after the moves).  With K = 0 the slot arrays
 * may be NULL (nothing moves).  No workspace. */
MOE_API moe_status taot_match_batched(const int32_t* expert_loads, const float* plan, int32_t B, int32_t E,
                              int32_t R, int32_t ranks_per_node, int32_t K,
                              int32_t* slot_expert, int32_t* slot_tokens, int32_t* rank_load,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Misc                                                                     */
/* ------------------------------------------------------------------------ */

/* Limit of every device-side wait (the grid barriers of the persistent
 * kernels), process-wide, in nanoseconds; 0 restores the default of 2 s.
 * When a wait expires, the kernel stops writing and returns, and the next
 * moe_get_device_status reports MOE_ERR_TIMEOUT.  Tests shorten the limit to
 * exercise that path; the library has no other use for it. */
MOE_API void moe_set_wait_timeout_ns(uint64_t ns);

/* Test hook for the timeout path, process-wide: with enable != 0 the grid
 * barriers of later launches wait for one CTA more than the grid holds, so no
 * barrier is ever released and every wait runs to its limit (shorten it with
 * moe_set_wait_timeout_ns first).  The kernels then stop writing after the
 * forward and return; moe_get_device_status reports MOE_ERR_TIMEOUT.  Nothing
 * faults or hangs.  0 restores normal barriers. */
MOE_API void moe_set_unreachable_barriers(int32_t enable);

/* Phase tracing of the persistent kernels (moe_router_fwd, moe_dispatch,
 * moe_router_step), process-wide.  With a non-NULL DEVICE buffer of
 * max_ctas * MOE_TRACE_POINTS uint64 values, every launch has CTA c write
 * %globaltimer (ns) to device_buf[c * MOE_TRACE_POINTS + i] at phase boundary
 * i (points a launch does not pass are left as they were):
 *   0 entry, 1 first forward ring stage landed, 2 forward rows done (warp 0),
 *   3 per-CTA partials published, 4 after the grid barrier, 5 totals, bases
 *   and offsets in shared memory, 6 (not recorded), 7 first backward stage available, 8 backward
 *   rows done (warp 0), 9 dispatch and E-sized outputs done (dispatch warp),
 *   10 all warps joined, 11 exit, 12 in-CTA dispatch ranks done (dispatch warp),
 *   13 the SM the CTA ran on (an SM id, not a time), 14 and 15 the time the
 *   last consumer warp finished its forward / backward rows. 
 * A launch with more than max_ctas CTAs fails with MOE_ERR_INVALID.  NULL
 * turns tracing off. */
#define MOE_TRACE_POINTS 16
MOE_API void moe_set_trace_buffer(uint64_t* device_buf, int32_t max_ctas);

MOE_API const char* moe_status_string(moe_status s);
MOE_API const char* moe_last_error(void);
MOE_API int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTER_H */
