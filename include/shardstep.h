/*
 * shardstep.h -- C ABI of libshardstep.so: the data-parallel hot path of a
 * ZeRO / FSDP sharded optimizer step over a FlatParameter, on one GPU.
 *
 * N_d data-parallel ranks are emulated as N_d buffers in one GPU's memory.
 * The reduce-scatter average, the AdamW update and the bf16 cast run as one
 * kernel pass; the all-gather is one copy kernel; packing and the DDP-style
 * bucketed all-reduce average are kernels of their own.
 *
 * Sources for what each call computes (page title, section / figure):
 *   [P1] "Infra: Data Parallel" (pufanyi.com blog)
 *   [P2] "PyTorch FSDP: 大模型分布式训练的工业级分片并行方案" (2048ai.net)
 *   [P3] "4.1 数据并行详解" (AIInfraGuide)
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are CUDA device addresses of the current device;
 *     "host" pointers are ordinary host memory.  Arrays *of* device pointers
 *     (src, grad_slices, shards, rank_grads) live in host memory.
 *   - The caller owns every buffer.  No entry point allocates or frees device
 *     memory, and none keeps a pointer after it returns.
 *   - Device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and is asynchronous: a zero return means the launch was
 *     accepted, not that the kernel has finished.  Kernel faults surface at
 *     the caller's next synchronisation, as usual in CUDA.
 *   - Arguments are validated on the host before anything is launched.  On
 *     error nothing is launched, a negative SHARDSTEP_ERR_* code is returned
 *     and shardstep_last_error() describes it (per calling thread).  Nothing is
 *     thrown across the ABI.
 *   - bf16 data is passed as uint16_t bit patterns.  fp32 arithmetic is IEEE
 *     single precision, round to nearest, with no contraction into fused
 *     multiply-adds, in the operation order each call states.
 *   - Every call is stateless and re-entrant; calls on different streams may
 *     run concurrently if their buffers do not overlap.
 *   - A call with no element to process (S = 0, n = 0, a unit whose tensors
 *     are all empty, no bucket or only empty buckets) launches nothing and
 *     returns SHARDSTEP_OK once its scalar arguments (nd, the sharding
 *     factor, the hyper-parameters or step state, the scaler's words) are
 *     valid; its data pointers are not looked at and may be NULL.
 */
#ifndef SHARDSTEP_H
#define SHARDSTEP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ codes */
#define SHARDSTEP_OK 0
#define SHARDSTEP_ERR_INVALID (-1)  /* bad pointer, size, dtype, rank or overlap */
#define SHARDSTEP_ERR_CUDA (-3)     /* the CUDA runtime refused a launch or query */
#define SHARDSTEP_ERR_TIMEOUT (-4)  /* a host-side wait ran past its limit */
#define SHARDSTEP_ERR_CAPACITY (-5) /* more ranks than SHARDSTEP_MAX_ND / a full buffer */
#define SHARDSTEP_ERR_IO (-6)       /* a checkpoint file could not be written or read back */

#define SHARDSTEP_DTYPE_BF16 0
#define SHARDSTEP_DTYPE_F32 1
#define SHARDSTEP_DTYPE_F16 2 /* IEEE half: gradients under fp16 loss scaling */

#define SHARDSTEP_MAX_ND 64 /* largest N_d a kernel accepts */

/* ------------------------------------------------------------ types */

/* AdamW hyper-parameters and the 1-based step count t.  The per-step fp32
 * scalars are derived on the host in double and rounded once to fp32:
 *   lr*wd, beta1, 1-beta1, beta2, 1-beta2, lr/bc1, sqrt(bc2), eps
 * with bc_i = 1 - beta_i^t, beta_i^t a left-to-right product of t factors. */
typedef struct {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    int64_t step;
} shardstep_adamw_t;

/* Sizes of a FlatParameter layout (see fsdp_layout). */
typedef struct {
    int64_t total;  /* T = sum of the tensors' numels             */
    int64_t padded; /* P = ceil(T / N_d) * N_d                     */
    int64_t shard;  /* S = P / N_d, elements per rank              */
    int32_t n_tensors;
    int32_t nd;
} shardstep_layout_info_t;

/* ------------------------------------------------------ FlatParameter */

/* fsdp_layout -- host only.
 * [P1] section "FSDP1：先打包，再切分" and its figure (FlatParameter of three
 * (4,2) weights on two ranks): the tensors of one FSDP unit are flattened and
 * concatenated in registration order, zero-padded at the tail to a multiple
 * of N_d, and split into N_d equal contiguous shards; a shard may cut a
 * tensor, and with use_orig_params a rank's view of a tensor it holds
 * nothing of is empty.
 *   numels[n]   host: elements of each tensor (>= 0), registration order.
 *   nd          N_d >= 1.
 *   info        host, required: T, P, S.
 *   offsets[n]  host or NULL: element offset of each tensor in the flat buffer.
 *   lo, hi      host or NULL, [nd * n], row r = rank: the piece of tensor t
 *               held by rank r is shard_r[lo[r*n+t], hi[r*n+t]) (shard
 *               coordinates, the tensor's overlap with [r*S, (r+1)*S) clamped
 *               to [0, S]); lo == hi when the rank holds nothing of it.
 * Errors: INVALID for n < 0, nd < 1, a negative numel, or a NULL array with
 * n > 0. */
int fsdp_layout(const int64_t* numels, int32_t n, int32_t nd, shardstep_layout_info_t* info,
                int64_t* offsets, int64_t* lo, int64_t* hi);

/* fsdp_flat_pack -- device.
 * Same source as fsdp_layout.  Writes flat[off_t + k] = src[t][k] for every
 * tensor t (a bit copy of contiguous row-major data) and flat[T..P) = 0.
 *   src[n]      host array of device pointers, one contiguous tensor each
 *               (may be NULL when numels[t] == 0).
 *   numels[n]   host, as in fsdp_layout.
 *   dtype       SHARDSTEP_DTYPE_BF16 (2-byte elements) or _F32 (4-byte).
 *   flat        device, P elements, must not overlap any source.
 * Any alignment is accepted; 16-byte-congruent source/destination pairs use
 * 16-byte accesses. */
int fsdp_flat_pack(const void* const* src, const int64_t* numels, int32_t n, int32_t nd,
                   int32_t dtype, void* flat, void* stream);

/* fsdp_shard_pieces -- host only.
 * Same source as fsdp_layout ([P1] "FSDP1：先打包，再切分": a shard may cut
 * a tensor, and a rank may hold nothing of one).  For rank `rank`, per
 * tensor t, where the piece of t that the rank holds sits on both sides:
 *   shard_lo[t]   its first position in the rank's shard (0..S),
 *   tensor_lo[t]  its first element within tensor t (row-major order),
 *   count[t]      its length (0 when the rank holds nothing of t; then
 *                 shard_lo and tensor_lo are 0),
 * so shard_r[shard_lo[t] + k] = tensor_t[tensor_lo[t] + k] for k < count[t]:
 * what a caller needs to fill a rank's shard from the original tensors, or
 * to write it back, without forming the full FlatParameter.
 *   numels[n]   host, as in fsdp_layout;  nd  N_d >= 1;  0 <= rank < nd.
 *   shard_lo, tensor_lo, count   host out, n entries each.
 * Errors: INVALID (as fsdp_layout, rank out of range, a NULL array). */
int fsdp_shard_pieces(const int64_t* numels, int32_t n, int32_t nd, int32_t rank,
                      int64_t* shard_lo, int64_t* tensor_lo, int64_t* count);

/* fsdp_views -- host only.
 * The use_orig_params views of [P1] section "FSDP1：先打包，再切分": per tensor,
 * the address and element count of its piece inside a buffer laid out by
 * fsdp_layout.  rank < 0: `base` is the full flat buffer of P elements (after
 * fsdp_ag_unpack), every tensor's view is whole and the padding is in none.
 * rank r >= 0: `base` is rank r's shard of S elements and each view is the
 * (possibly empty) piece the rank holds; an empty view has count 0 and the
 * address of shard position lo.
 *   elem_size   bytes per element (2 or 4).
 *   ptrs[n], counts[n]  host outputs. */
int fsdp_views(const int64_t* numels, int32_t n, int32_t nd, int32_t rank, void* base,
               int32_t elem_size, void** ptrs, int64_t* counts);

/* ----------------------------------------------------- accumulation */

/* fsdp_grad_accumulate -- device.
 * [P1] section "Naïve Data Parallelism": with gradient accumulation over M
 * micro-batches the gradients are summed locally and only the last
 * micro-batch synchronises; each micro-batch loss is divided by M, which
 * scales its gradient by 1/M.  Per element, in fp32:
 *     first != 0:  acc[i] = g[i] * scale
 *     first == 0:  acc[i] = acc[i] + g[i] * scale
 * where g is upcast from bf16 exactly and `scale` is the fp32 value of 1/M.
 *   g     device, n bf16.      acc  device, n fp32 (read unless first).
 * g and acc must not overlap. */
int fsdp_grad_accumulate(const uint16_t* g, float* acc, int64_t n, float scale, int32_t first,
                         void* stream);

/* ------------------------------------------------- the fused step */

/* fsdp_rs_avg_adamw_cast -- device, one kernel pass.
 * Rank r's part of a ZeRO / FSDP optimizer step: [P1] ZeRO section (reduce-
 * scatter with averaging hands each rank its part of the averaged gradient;
 * AdamW is elementwise so the rank updates only its shard and its moments);
 * [P3] section 2 (the mean of the N_d local-mean gradients is the global
 * gradient); [P2] section 3.5 (one high-to-low cast; communication in low
 * precision, so the cast precedes the all-gather).  Per shard element i:
 *     g  = (((G_0[i] + G_1[i]) + G_2[i]) + ... + G_{N_d-1}[i]) / N_d
 *          (fp32, rank order; G_q upcast exactly from bf16, or fp32 when
 *           micro-batches were accumulated; a power-of-two N_d multiplies by
 *           the exact reciprocal, which gives the same result)
 *     p  = p - (lr*wd) * p
 *     m  = beta1 * m + (1-beta1) * g
 *     v  = beta2 * v + ((1-beta2) * g) * g
 *     p  = p - ((lr/bc1) * m) / (sqrt(v) / sqrt(bc2) + eps)
 *     out[i] = bf16(p), round to nearest even
 *   grad_slices[nd]  host array of device pointers: grad_slices[q] is rank
 *                    q's contribution to this rank's shard, S elements of
 *                    grad_dtype (i.e. rank q's flat gradient + r*S).
 *   grad_dtype       SHARDSTEP_DTYPE_BF16, _F32 or _F16 (upcast exactly).
 *   nd               1 <= N_d <= SHARDSTEP_MAX_ND (N_d = 1 is a plain,
 *                    unsharded AdamW + cast over S elements).
 *   master, m, v     device, S fp32 each, updated in place.
 *   out_bf16         device, S bf16; may be the rank's slot of the full flat
 *                    parameter buffer (full + r*S).
 * The gradient inputs must not overlap any output; master, m, v and out_bf16
 * must not overlap one another.  Any alignment is accepted.  Kernels:
 * (1) register-staged, 4 elements per access -- needs state 16-byte, bf16
 * slices and out 8-byte, fp32 slices 16-byte alignment; the default where
 * N_d is 1 to 8, 12 or 16 (5, 7, 12 and 16 not with fp32 slices), and where
 * two TMA stages do not fit; (2) TMA-staged --
 * needs S >= 4096, master / m / v and every slice 16-byte aligned, out_bf16
 * 8-byte aligned, and two stages of 2048 x (N_d x grad bytes + 12) bytes
 * within the per-block shared-memory limit (N_d <= 22 for bf16, <= 11 for
 * fp32 on GB300); the default for other N_d >= 3; (3) one element per
 * access.  All three compute the same bits.  A TMA-staged launch whose
 * internal wait runs out (about 2 s) sets a bit in the device status word;
 * see shardstep_device_status.
 * Errors: INVALID (null pointer, S < 0, step < 1, bad dtype, overlap),
 * CAPACITY (nd > SHARDSTEP_MAX_ND), CUDA (launch refused). */
int fsdp_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                           int64_t S, float* master, float* m, float* v, uint16_t* out_bf16,
                           const shardstep_adamw_t* hp, void* stream);

/* fsdp_accumulate_rs_avg_adamw_cast -- device, one kernel pass.
 * The last of M micro-batches ([P1] section "Naïve Data Parallelism": the
 * gradients accumulate locally and only the last micro-batch synchronises)
 * accumulated and reduce-scattered in the same pass.  Rank q's contribution
 * to this rank's shard is the value fsdp_grad_accumulate(first = 0) would
 * store for the last micro-batch,
 *     G_q[i] = acc_slices[q][i] + bf16->fp32(last_slices[q][i]) * scale
 * (fp32, the product rounded, then the sum), and the step proceeds exactly
 * as fsdp_rs_avg_adamw_cast with fp32 slices G_q: the same bits as
 * fsdp_grad_accumulate on every rank's slice followed by the fused step.
 * The accumulators are read, not written: afterwards they still hold
 * micro-batches 0..M-2.  Per shard element it moves 6*N_d + 26 bytes where
 * the two calls move 14*N_d + 26.
 *   acc_slices[nd]   host array of device pointers: rank q's fp32
 *                    accumulator (micro-batches 0..M-2) + r*S, S elements.
 *   last_slices[nd]  host array of device pointers: rank q's bf16 gradient
 *                    of the last micro-batch + r*S, S elements.
 *   shard_group      F: nd for plain sharding (rank-order sum), else the
 *                    sharding factor of hybrid sharding, summed in the order
 *                    of fsdp_hybrid_rs_avg_adamw_cast (F must divide nd).
 *   scale            the fp32 value of 1/M, as given to fsdp_grad_accumulate.
 *   nd, S, master, m, v, out_bf16, hp: as in fsdp_rs_avg_adamw_cast.
 * No input slice may overlap an output; the outputs must not overlap one
 * another.  Any alignment is accepted; accumulator slices and state 16-byte
 * aligned with bf16 slices and out_bf16 8-byte aligned take the vector
 * kernel (4 elements per access), anything else one element per access.
 * Errors: INVALID (null pointer, S < 0, step < 1, overlap, a shard_group
 * that does not divide nd), CAPACITY (nd > SHARDSTEP_MAX_ND), CUDA (launch
 * refused). */
int fsdp_accumulate_rs_avg_adamw_cast(const float* const* acc_slices,
                                      const uint16_t* const* last_slices, int32_t nd,
                                      int32_t shard_group, int64_t S, float scale, float* master,
                                      float* m, float* v, uint16_t* out_bf16,
                                      const shardstep_adamw_t* hp, void* stream);

/* fsdp_hybrid_rs_avg_adamw_cast -- device, one kernel pass.
 * Hybrid sharding with sharding factor F = shard_group ([P2] section 2,
 * sharding factor: F = 1 is full replication, F = N_d full sharding; [P2]
 * section 3.3: full sharding inside groups of F GPUs, replication across the
 * groups; [P3] section 6.3, HYBRID_SHARD).  The N_d = R x F ranks are ordered
 * k = g*F + j (group g, position j); a unit is split into F shards of S
 * elements and rank (g, f) holds shard f, replicated in each of the R groups.
 * Its gradient is reduce-scattered inside its group, all-reduced across the
 * groups and averaged over all N_d ranks; per element, in fp32:
 *     s_g = G_{gF} + G_{gF+1} + ... + G_{gF+F-1}        (order j)
 *     g   = (s_0 + s_1 + ... + s_{R-1}) / N_d            (order g)
 * followed by the same AdamW update and bf16 cast as fsdp_rs_avg_adamw_cast.
 * shard_group = nd gives exactly fsdp_rs_avg_adamw_cast; shard_group = 1 the
 * plain all-reduce average of every rank.
 *   grad_slices[nd]  rank k's contribution to shard f (S elements each), in
 *                    rank order k = g*F + j.
 *   shard_group      F >= 1, dividing nd.
 * Other arguments, aliasing rules, kernel choice and errors as in
 * fsdp_rs_avg_adamw_cast; INVALID when F does not divide nd. */
int fsdp_hybrid_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                  int32_t shard_group, int64_t S, float* master, float* m,
                                  float* v, uint16_t* out_bf16, const shardstep_adamw_t* hp,
                                  void* stream);

/* ---------------------------------------- device-resident step count */

/* AdamW step state kept in device memory, so that a training step needs no
 * host work: the advance, the fused update and the all-gather can be
 * captured once in a CUDA graph and replayed every iteration.  The caller
 * allocates it (device memory, 8-byte aligned, sizeof 56 bytes); the fields
 * are written only by the calls below.  The per-step scalars are derived as
 * the host-scalar entry points derive them, so both give the same bits:
 * beta^t is the running product of t factors in double, then 1 - beta^t,
 * lr / (1 - beta1^t), sqrt(1 - beta2^t), lr * wd, 1 - beta, each in double
 * and rounded once to fp32 (the host does the same from hp->step). */
typedef struct {
    int64_t step;         /* t of the scalars below; 0 = none yet          */
    double beta1_pow;     /* beta1^t                                        */
    double beta2_pow;     /* beta2^t                                        */
    float scalars[8];     /* fp32 scalars of step t (layout internal)       */
} shardstep_adamw_state_t;

/* shardstep_adamw_state_init -- device, one thread.  Sets *state to step
 * `step` >= 0 of hp's betas (the powers from the host's running product);
 * for step >= 1 also that step's scalars, so a state restored at the step of
 * a checkpoint continues exactly.  hp->step is ignored.  Asynchronous on
 * `stream`.  Errors: INVALID (null or misaligned state, null hp, step < 0),
 * CUDA. */
int shardstep_adamw_state_init(shardstep_adamw_state_t* state, const shardstep_adamw_t* hp,
                               int64_t step, void* stream);

/* shardstep_adamw_state_advance -- device, one thread.  Moves *state from
 * step t to t + 1 (beta powers times the betas) and derives the scalars of
 * step t + 1 from hp's lr, betas, eps and weight decay, which the call
 * passes by value (a captured graph replays the values it was captured
 * with).  hp->step is ignored.
 *   skip   NULL, or a device word: when it holds a non-zero value as the
 *          kernel runs, the state is left unchanged -- pass the gradient
 *          scaler's found_inf so that a skipped step does not count, as an
 *          optimizer step that the scaler skips does not.
 * Errors as shardstep_adamw_state_init, and INVALID for a misaligned skip. */
int shardstep_adamw_state_advance(shardstep_adamw_state_t* state, const shardstep_adamw_t* hp,
                                  const uint32_t* skip, void* stream);

/* fsdp_state_rs_avg_adamw_cast -- device, one kernel pass.  The fused step
 * of fsdp_hybrid_rs_avg_adamw_cast (shard_group = nd: of
 * fsdp_rs_avg_adamw_cast) with the AdamW scalars read on the device from
 * *state, which must hold a step >= 1 (an advance or an init with step >= 1
 * before it in stream order); the result is bit-identical to the host-scalar
 * call at hp->step = state->step.  The call does no host work that depends
 * on the step, so it can be captured in a CUDA graph.  Other arguments,
 * aliasing rules, kernel choice and errors as in
 * fsdp_hybrid_rs_avg_adamw_cast; INVALID for a null or misaligned state. */
int fsdp_state_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                 int32_t shard_group, int64_t S, float* master, float* m,
                                 float* v, uint16_t* out_bf16,
                                 const shardstep_adamw_state_t* state, void* stream);

/* fsdp_state_accumulate_rs_avg_adamw_cast -- device, one kernel pass.
 * fsdp_accumulate_rs_avg_adamw_cast with the AdamW scalars read on the device
 * from a step state (shardstep_adamw_state_init / _advance), so that the
 * call launches the same kernel with the same arguments every step and can
 * be captured in a CUDA graph.  `state`: device, 8-byte aligned, at a step
 * >= 1 (advance it before the call).  Errors: those of
 * fsdp_accumulate_rs_avg_adamw_cast, and INVALID for a NULL or misaligned
 * state. */
int fsdp_state_accumulate_rs_avg_adamw_cast(const float* const* acc_slices,
                                            const uint16_t* const* last_slices, int32_t nd,
                                            int32_t shard_group, int64_t S, float scale,
                                            float* master, float* m, float* v,
                                            uint16_t* out_bf16,
                                            const shardstep_adamw_state_t* state,
                                            void* stream);

/* ------------------------------------------------ gradient scaler */

/* Sharded gradient scaler for fp16 loss scaling ([P2] section 3.5: a sharded
 * gradient scaler adapted to parameter sharding keeps gradient scaling
 * mathematically equivalent; the page gives no mechanism).  Reading: the loss
 * is multiplied by a scale s, so the fp16 gradients (SHARDSTEP_DTYPE_F16)
 * arrive multiplied by s; each rank multiplies its reduced shard gradient by
 * 1/s and checks it for inf / NaN; the flags are OR-ed over all ranks (one
 * shared device word: calling the check for every rank's shard is the
 * all-reduce); a flagged step changes no parameter, moment or bf16 output on
 * any rank; the scale then backs off, or grows after growth_interval clean
 * steps.  One step:
 *     fsdp_grad_unscale_check(rank r's slices ...)      for every rank r
 *     fsdp_scaled_rs_avg_adamw_cast(rank r ...)          for every rank r
 *     fsdp_grad_scaler_update(...)                       once
 *
 * The scale lives in a device word the caller owns (read, never written, by
 * the check and the step; written by the update), so a step needs no
 * host-side knowledge of it: each kernel computes inv = fl32(1 / *scale).
 *
 * fsdp_grad_unscale_check -- device.  Sets *found_inf to 1 when any element
 * of g = fl(reduced mean of the slices * inv) (the reduce in the order of
 * fsdp_hybrid_rs_avg_adamw_cast; shard_group = nd is the plain rank order)
 * is inf or NaN; never clears it.  Reads the slices only.
 *   scale      device, one fp32 word: the current loss scale s.
 *   found_inf  device, one 4-byte word, zero at the start of the step. */
int fsdp_grad_unscale_check(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                            int32_t shard_group, int64_t S, const float* scale,
                            uint32_t* found_inf, void* stream);

/* fsdp_state_scaled_rs_avg_adamw_cast -- device, one kernel pass.  The step
 * of fsdp_scaled_rs_avg_adamw_cast (unscaled by 1 / *scale, skipped when
 * *found_inf is non-zero) with the AdamW scalars read from *state, as in
 * fsdp_state_rs_avg_adamw_cast.  With the check before it, an advance
 * whose skip word is found_inf and fsdp_grad_scaler_update after it, the
 * whole loss-scaled step runs from device words and can be captured in a
 * CUDA graph.  Arguments and errors as fsdp_scaled_rs_avg_adamw_cast, with
 * state in place of hp. */
int fsdp_state_scaled_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype,
                                        int32_t nd, int32_t shard_group, int64_t S,
                                        float* master, float* m, float* v, uint16_t* out_bf16,
                                        const shardstep_adamw_state_t* state, const float* scale,
                                        const uint32_t* found_inf, void* stream);

/* fsdp_scaled_rs_avg_adamw_cast -- device, one kernel pass.  The fused step
 * of fsdp_hybrid_rs_avg_adamw_cast on the unscaled gradient
 *     g = fl(reduced mean * fl32(1 / *scale))
 * when *found_inf is 0 at launch; when it is non-zero every CTA returns at
 * once and nothing is written.  Other arguments as
 * fsdp_hybrid_rs_avg_adamw_cast. */
int fsdp_scaled_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                  int32_t shard_group, int64_t S, float* master, float* m,
                                  float* v, uint16_t* out_bf16, const shardstep_adamw_t* hp,
                                  const float* scale, const uint32_t* found_inf, void* stream);

/* fsdp_grad_scaler_update -- device, one thread.  fp32 arithmetic:
 *     found:  scale = scale * backoff_factor, growth_tracker = 0
 *     else:   growth_tracker += 1; when it reaches growth_interval the scale
 *             becomes scale * growth_factor if that is finite, and the
 *             tracker returns to 0
 * then *found_inf = 0 for the next step.  All three are device words
 * (float, int32, uint32) the caller owns.  INVALID for NULL or
 * growth_interval < 1. */
int fsdp_grad_scaler_update(float* scale, int32_t* growth_tracker, uint32_t* found_inf,
                            float growth_factor, float backoff_factor, int32_t growth_interval,
                            void* stream);

/* ------------------------------------------------------ all-gather */

/* fsdp_ag_unpack -- device, one kernel.
 * [P1] ZeRO section and [P2] section 3.1: after the update each rank's bf16
 * shard is all-gathered so every rank holds the whole unit again; [P3]
 * section 5.1: all-gather concatenates the per-rank pieces.
 *     full[q*S + i] = shards[q][i]     for q < N_d, i < S
 * Use fsdp_views(rank = -1) for the per-tensor views of `full`.
 *   shards[nd]  host array of device pointers, S bf16 each.  shards[q] may
 *               equal full + q*S (that copy is skipped); otherwise no shard
 *               may overlap `full`.
 *   full        device, nd*S bf16. */
int fsdp_ag_unpack(const uint16_t* const* shards, int32_t nd, int64_t S, uint16_t* full,
                   void* stream);

/* ---------------------------------------------------------- FSDP2 */

/* FSDP2 per-parameter sharding along dim 0 ([P1] section "FSDP2：分别记录每个
 * 参数的分片" and its figure: each parameter of a fully_shard group is split
 * along dim 0 -- a (4,2) weight on two ranks is (2,2) locally, an (8,4)
 * weight on four ranks (2,4) -- while the group is still communicated with
 * one all-gather and one reduce-scatter).  Parameter t has dim0[t] rows of
 * row[t] elements (row = product of the trailing dims, 1 for a vector).
 * Rank r holds rows [r*c_t, min((r+1)*c_t, dim0[t])), c_t = ceil(dim0[t] /
 * nd), possibly none.  A rank's local buffer of the group concatenates, in
 * registration order, its rows of every parameter zero-padded to c_t rows:
 * local = sum_t c_t * row[t] elements; parameter t starts at offset[t].  The
 * group's communication buffers are rank-major: nd pieces of `local`.
 *
 * fsdp2_layout -- host only: chunk[n] (c_t), offset[n] (may be NULL) and
 * *local.  Errors: INVALID for n < 0, nd < 1, negative sizes, NULL arrays. */
int fsdp2_layout(const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd, int64_t* chunk,
                 int64_t* offset, int64_t* local);

/* fsdp2_local_views -- host only: DTensor.to_local() of rank `rank` inside its
 * local buffer `base`: ptrs[t] = base + offset[t] elements, rows[t] = the
 * rows it holds (the local shape is (rows[t], trailing dims)). */
int fsdp2_local_views(const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd,
                      int32_t rank, void* base, int32_t elem_size, void** ptrs, int64_t* rows);

/* fsdp2_chunk_cat -- device, batched copy.  One rank's reduce-scatter input:
 *     out[r*local + offset[t] + k] = grads[t][r*c_t*row[t] + k]   (held rows)
 *                                  = 0                             (padding rows)
 * for every rank piece r and parameter t, so that
 * fsdp_rs_avg_adamw_cast over the N_d ranks' buffers (slices at r*local)
 * reduce-scatters the group.
 *   grads[n]  host array of device pointers, full contiguous tensors.
 *   out       device, nd*local elements, must not overlap any gradient.
 *   dtype     SHARDSTEP_DTYPE_BF16 or _F32. */
int fsdp2_chunk_cat(const void* const* grads, const int64_t* dim0, const int64_t* row, int32_t n,
                    int32_t nd, int32_t dtype, void* out, void* stream);

/* fsdp2_all_gather_copy_out -- device, batched copy.  All-gather of the ranks'
 * local buffers straight into the full per-parameter tensors (no
 * intermediate gather buffer):
 *     params[t][r*c_t*row[t] + k] = local_bufs[r][offset[t] + k]   (held rows)
 *   local_bufs[nd]  host array of device pointers, `local` elements each.
 *   params[n]       host array of device pointers, full contiguous tensors of
 *                   dim0[t]*row[t] elements; must not overlap the buffers. */
int fsdp2_all_gather_copy_out(const void* const* local_bufs, const int64_t* dim0,
                              const int64_t* row, int32_t n, int32_t nd, int32_t dtype,
                              void* const* params, void* stream);

/* fsdp2_rs_avg_adamw_cast -- device; one fused launch per parameter the rank
 * holds rows of, one small launch per parameter with padding rows.
 * Rank `rank`'s FSDP2 optimizer step read straight from the ranks' full
 * per-parameter gradients ([P1] FSDP2 section: a group's parameters are
 * reduce-scattered together; the emulated reduce-scatter needs no
 * contiguous send buffer, so the chunk-cat copy is skipped).  The same bits
 * as fsdp2_chunk_cat of every rank's gradients followed by
 * fsdp_rs_avg_adamw_cast over the N_d pieces at rank*local: at held rows
 *     g = (grads[0][t][j] + grads[1][t][j] + ...) / N_d,
 *     j = rank*c_t*row[t] + k   (rank order, fp32, as fsdp_rs_avg_adamw_cast)
 * and at padding rows every contribution is +0, so AdamW runs on g = +0.
 *   grads[nd*n]   host array of device pointers: grads[q*n + t] is rank q's
 *                 full contiguous gradient of parameter t (dim0[t]*row[t]
 *                 elements; NULL allowed for an empty parameter), all of
 *                 grad_dtype (SHARDSTEP_DTYPE_BF16, _F16 or _F32).
 *   dim0, row, n  the group's shapes, as in fsdp2_layout.
 *   rank          0 <= rank < nd.
 *   master, m, v  device fp32, the rank's padded local buffers (`local`
 *                 elements, fsdp2_layout's offsets), updated in place.
 *   out_bf16      device, `local` elements: the updated parameters in bf16.
 *   hp            host, as in fsdp_rs_avg_adamw_cast.
 * No gradient may overlap an output; the outputs must not overlap one
 * another.  Errors: INVALID (dtype, nd, rank, NULL, alignment, overlap, bad
 * shapes), CAPACITY (nd > SHARDSTEP_MAX_ND), CUDA. */
int fsdp2_rs_avg_adamw_cast(const void* const* grads, int32_t grad_dtype, const int64_t* dim0,
                            const int64_t* row, int32_t n, int32_t nd, int32_t rank,
                            float* master, float* m, float* v, uint16_t* out_bf16,
                            const shardstep_adamw_t* hp, void* stream);

/* fsdp2_state_rs_avg_adamw_cast -- device; fsdp2_rs_avg_adamw_cast with the
 * AdamW scalars read on the device from `state` (at a step >= 1; see
 * shardstep_adamw_state_t), so that the FSDP2 step of every rank can be
 * captured in a CUDA graph with shardstep_adamw_state_advance before it.
 * Same bits as the host-scalar call at the state's step. */
int fsdp2_state_rs_avg_adamw_cast(const void* const* grads, int32_t grad_dtype,
                                  const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd,
                                  int32_t rank, float* master, float* m, float* v,
                                  uint16_t* out_bf16, const shardstep_adamw_state_t* state,
                                  void* stream);

/* ---------------------------------------------------- DDP buckets */

/* ddp_bucket_plan -- host only.
 * [P3] section 4.2: gradients are grouped into buckets in the order backward
 * produces them (reverse registration order), capped at bucket_cap_mb
 * (~25 MB by default).  Rule used: walk the parameters in reverse order; close
 * the open bucket before a parameter that would take it past cap_bytes; a
 * parameter larger than the cap gets a bucket of its own; parameters are never
 * split; zero-size parameters join the open bucket.
 *   numels[n]          host, registration order.
 *   elem_size          bytes per gradient element (> 0).
 *   cap_bytes          > 0.
 *   param_offset[n]    host out: element offset of each parameter in the
 *                      bucketed flat buffer (buckets back to back).
 *   bucket_of_param[n] host out.
 *   bucket_offsets     host out, n + 1 entries available; the first
 *                      n_buckets + 1 are the buckets' element offsets.
 *   n_buckets          host out. */
int ddp_bucket_plan(const int64_t* numels, int32_t n, int32_t elem_size, int64_t cap_bytes,
                    int64_t* param_offset, int32_t* bucket_of_param, int64_t* bucket_offsets,
                    int32_t* n_buckets);

/* ddp_bucket_allreduce_avg -- device, one launch per bucket.
 * [P1] section "Naïve Data Parallelism" and [P3] section 4.2: each bucket's
 * gradients are all-reduce-averaged over the N_d ranks; the all-reduce keeps
 * the bf16 dtype, so for every element k of buckets first..first+count-1:
 *     out[k] = bf16((((G_0[k] + G_1[k]) + ...) + G_{N_d-1}[k]) / N_d)
 * with the sum in fp32, rank order.  Follow with fsdp_rs_avg_adamw_cast at
 * nd = 1 on the averaged gradient for the replicated (unsharded) update.
 *   rank_grads[nd]     host array of device pointers, bucketed flat gradient
 *                      of each rank (bf16).
 *   bucket_offsets     host, element offsets from ddp_bucket_plan.
 *   first, count       the buckets to reduce (a bucket is reduced as soon as
 *                      it is ready, so callers may go bucket by bucket).
 *   out                device bf16, same indexing as the rank buffers; must
 *                      not overlap them. */
int ddp_bucket_allreduce_avg(const uint16_t* const* rank_grads, int32_t nd,
                             const int64_t* bucket_offsets, int32_t first, int32_t count,
                             uint16_t* out, void* stream);

/* ddp_bucket_allreduce_avg_adamw_cast -- device, one launch.
 * The same sources as ddp_bucket_allreduce_avg, with the replicated update
 * that follows it in one pass ([P1] section "Naïve Data Parallelism": every
 * rank averages the full gradient and runs the same optimizer step).  For
 * every element k of buckets first..first+count-1 (one contiguous range):
 *     h        = bf16((((G_0[k] + G_1[k]) + ...) + G_{N_d-1}[k]) / N_d)
 *                (fp32 sum in rank order; the all-reduce keeps bf16)
 *     mean_out[k] = h                      (when mean_out is not NULL)
 *     master[k], m[k], v[k], params[k]     AdamW of fsdp_rs_avg_adamw_cast
 *                with g = bf16->fp32(h), then params[k] = bf16(master[k])
 * i.e. the bits of ddp_bucket_allreduce_avg followed by
 * fsdp_rs_avg_adamw_cast at nd = 1 on its output, without writing the mean
 * and reading it back (2 N_d + 26 bytes per element instead of
 * 2 N_d + 2 + 28; + 2 when mean_out is kept).
 *   rank_grads[nd]   host array of device pointers, as in
 *                    ddp_bucket_allreduce_avg (bf16).
 *   bucket_offsets   host, from ddp_bucket_plan; first, count as there.
 *   mean_out         device bf16 or NULL (the averaged gradient is not kept).
 *   master, m, v     device fp32, params device bf16: the replicated state,
 *                    indexed like the rank buffers (bucketed flat order),
 *                    updated in place over the buckets' range.
 *   hp               AdamW hyper-parameters and step t >= 1.
 * The outputs must not overlap one another or any gradient.  Any alignment
 * is accepted (4-element accesses need the state 16-byte, the gradients,
 * mean_out and params 8-byte aligned at the range's start).  Register-staged
 * kernels only.
 * Errors: INVALID (null pointer, decreasing offsets, step < 1, overlap),
 * CAPACITY (nd > SHARDSTEP_MAX_ND), CUDA (launch refused). */
int ddp_bucket_allreduce_avg_adamw_cast(const uint16_t* const* rank_grads, int32_t nd,
                                        const int64_t* bucket_offsets, int32_t first,
                                        int32_t count, uint16_t* mean_out, float* master,
                                        float* m, float* v, uint16_t* params,
                                        const shardstep_adamw_t* hp, void* stream);

/* ---------------------------------------------- DDP bucket readiness
 * Host only.  [P3] section 4.2: a bucket is all-reduced as soon as every
 * gradient in it is ready, so the buckets' reductions overlap the rest of
 * backward; [P3] section 4.2 also names the failure: a parameter that the
 * forward pass did not use never gets a gradient, its bucket never fills and
 * the all-reduce waits forever (the case find_unused_parameters covers).
 * Reading: the N_d emulated ranks (host threads) mark each parameter's
 * gradient ready; a caller waits for a bucket on the host with a limit and
 * launches its all-reduce only when every rank has marked every parameter
 * in it.  A wait that runs out returns TIMEOUT and names one missing
 * (rank, parameter); no kernel is launched for the bucket and nothing waits
 * on the GPU.  The table lives in caller-provided host memory of
 * ddp_ready_bytes() bytes, 8-byte aligned; marks from several threads are
 * atomic; a wait may run concurrently with marks. */

/* Bytes of the table for n_params parameters in n_buckets buckets and nd
 * ranks; -1 for invalid sizes. */
int64_t ddp_ready_bytes(int32_t n_params, int32_t n_buckets, int32_t nd);

/* Sets up the table: bucket_of_param[n_params] (host, from ddp_bucket_plan)
 * gives each parameter's bucket; every (rank, parameter) starts unmarked.
 * Errors: INVALID (NULL, misaligned, bucket index out of range), CAPACITY
 * (table_bytes too small). */
int ddp_ready_init(void* table, int64_t table_bytes, const int32_t* bucket_of_param,
                   int32_t n_params, int32_t n_buckets, int32_t nd);

/* Rank `rank` has the gradient of parameter `param` in device memory: mark
 * only after the writes that produced it have completed (the bucket's
 * all-reduce may be launched on another stream as soon as this mark
 * completes the bucket; the table orders host threads, not device work).
 * *bucket_done (may be NULL) receives the bucket this mark completed on all
 * ranks, else -1.
 * Errors: INVALID (uninitialised table, out of range, marked twice). */
int ddp_ready_mark(void* table, int32_t rank, int32_t param, int32_t* bucket_done);

/* Waits up to timeout_us microseconds (host, sleeping between checks) until
 * every rank has marked every parameter of `bucket`.  OK when it has;
 * TIMEOUT otherwise, with *missing_rank / *missing_param (either may be NULL)
 * naming one (rank, parameter) that never arrived (-1 when ready).  Errors:
 * INVALID. */
int ddp_ready_wait(void* table, int32_t bucket, int64_t timeout_us, int32_t* missing_rank,
                   int32_t* missing_param);

/* Unmarks everything for the next iteration (no marks or waits may run
 * concurrently).  Errors: INVALID. */
int ddp_ready_reset(void* table);

/* --------------------------------------------------------- ledger */

/* Model-state bytes per GPU ([P1] ZeRO figure; [P3] section 7), 16-bit
 * parameters and gradients, k bytes of optimizer state per parameter:
 *   stage 0: 2Ψ + 2Ψ + kΨ          stage 1: 2Ψ + 2Ψ + kΨ/N_d
 *   stage 2: 2Ψ + (2Ψ + kΨ)/N_d    stage 3: (2Ψ + 2Ψ + kΨ)/N_d
 * Returns a negative value for a bad stage or nd < 1. */
double shardstep_state_bytes(double psi, int32_t nd, int32_t stage, double k);

/* Bytes sent per GPU for one step's communication ([P1] ZeRO section; [P3]
 * sections 5 and 8), ring model, 16-bit elements; `exact` keeps the
 * (N_d-1)/N_d factor the pages drop. */
#define SHARDSTEP_COMM_REDUCE_SCATTER 0 /* 2Ψ                  */
#define SHARDSTEP_COMM_ALL_GATHER 1     /* 2Ψ                  */
#define SHARDSTEP_COMM_ALL_REDUCE 2     /* 4Ψ (naive DP / DDP) */
#define SHARDSTEP_COMM_ZERO1 3          /* 4Ψ                  */
#define SHARDSTEP_COMM_ZERO2 4          /* 4Ψ                  */
#define SHARDSTEP_COMM_ZERO3 5          /* 6Ψ                  */
double shardstep_comm_bytes(double psi, int32_t nd, int32_t kind, int32_t exact);

/* Hybrid sharding ledger ([P2] section 3.3): model-state bytes per GPU are
 * the ZeRO-3 ledger with N_d replaced by F, (2Ψ + 2Ψ + kΨ)/F; per-GPU bytes
 * sent per step, ring model, 16-bit elements (exact keeps the (n-1)/n
 * factors):
 *   SHARDSTEP_HYBRID_INTRA  reduce-scatter + all-gather inside the group of F:
 *                           2 x 2Ψ (F-1)/F
 *   SHARDSTEP_HYBRID_INTER  all-reduce of the GPU's Ψ/F shard across the
 *                           R = N_d/F groups: 4 (Ψ/F) (R-1)/R
 * Both return a negative value when F < 1 or F does not divide nd. */
#define SHARDSTEP_HYBRID_INTRA 0
#define SHARDSTEP_HYBRID_INTER 1
double shardstep_hybrid_state_bytes(double psi, int32_t shard_group, double k);
double shardstep_hybrid_comm_bytes(double psi, int32_t nd, int32_t shard_group, int32_t kind,
                                   int32_t exact);

/* ----------------------------------------------------- checkpoint */

/* Sharded checkpoint ([P1] section "Checkpoint：让各张卡保存自己的分片": with
 * the model state spread over the GPUs, each rank saves the shards it owns
 * and the metadata needed to restore them; a load reads according to the
 * target sharding layout, so the rank count may change between saving and
 * loading; optimizer state is saved with the weights).  Host only: the
 * caller stages device state through host memory.
 *
 * A rank file holds a 64-byte header (magic "SHSTCKPT", version 2, nd, rank,
 * section count, step, the tables' checksum), the element count T_u of
 * every unit's FlatParameter, a section table and the sections, each at a
 * 4096-byte aligned offset with its checksum.  Checksums are FNV-1a
 * (64-bit) over little-endian 64-bit words, a trailing partial word
 * zero-padded: the tables' one chain; a section's four chains, word j in
 * chain j mod 4, whose four values are then folded in chain order by one
 * more chain (version 1 files, whose sections have one chain, are read and
 * verified too).  It is written to "<path>.tmp" and renamed into place. */
typedef struct {
    int32_t unit;     /* unit index, 0 <= unit < n_units        */
    int32_t kind;     /* caller's tag, e.g. 0 master, 1 m, 2 v  */
    int64_t bytes;
    const void* data; /* host memory                            */
} shardstep_ckpt_section_t;

typedef struct {
    int32_t nd, rank, n_units, n_sections;
    int64_t step;
} shardstep_ckpt_info_t;

/* One piece of a reshard plan, in elements of a unit's FlatParameter. */
typedef struct {
    int32_t old_rank;   /* saved rank file to read                 */
    int32_t pad_;
    int64_t old_offset; /* element offset in that rank's shard     */
    int64_t new_offset; /* element offset in the new rank's shard  */
    int64_t count;
} shardstep_ckpt_piece_t;

/* Writes rank `rank`'s file of a checkpoint taken with nd ranks.
 * Errors: INVALID (arguments), IO (create / write / rename failed). */
int shardstep_ckpt_save_rank(const char* path, int32_t nd, int32_t rank, int64_t step,
                             const int64_t* unit_totals, int32_t n_units,
                             const shardstep_ckpt_section_t* sections, int32_t n_sections);

/* Header of a rank file; unit_totals (may be NULL) receives up to cap_units
 * unit element counts.  The tables' checksum is verified.  Errors: IO. */
int shardstep_ckpt_info(const char* path, shardstep_ckpt_info_t* info, int64_t* unit_totals,
                        int32_t cap_units);

/* Reads `bytes` bytes at `byte_offset` of the section (unit, kind) into dst
 * (host).  Errors: INVALID (no such section, range outside it), IO. */
int shardstep_ckpt_read(const char* path, int32_t unit, int32_t kind, int64_t byte_offset,
                        int64_t bytes, void* dst);

/* Reads every section of a rank file and checks its checksum.  Errors: IO
 * on the first mismatch. */
int shardstep_ckpt_verify(const char* path);

/* The pieces of the saved shards (old_nd ranks, FlatParameter layout of a
 * unit of `total` elements) that make up rank new_rank's shard under new_nd
 * ranks, in new-offset order; positions at or past `total` are padding (zero)
 * and in no piece.  pieces[cap]; *n_pieces receives the count (CAPACITY when
 * it exceeds cap). */
int fsdp_reshard_plan(int64_t total, int32_t old_nd, int32_t new_nd, int32_t new_rank,
                      shardstep_ckpt_piece_t* pieces, int32_t cap, int32_t* n_pieces);

/* ------------------------------------------------------------ misc */

/* Selects the kernels the streaming calls may use, process-wide: the fused
 * steps (plain, hybrid, scaled), fsdp_grad_accumulate,
 * ddp_bucket_allreduce_avg and fsdp_grad_unscale_check.
 * SHARDSTEP_PATH_TMA uses the TMA-staged kernels whenever the arguments
 * allow it (every source 16-byte aligned, at least 4096 elements, two stages
 * in shared memory); _REGISTER uses only the register-staged kernels;
 * _AUTO (default) uses the TMA-staged kernels where they measured faster:
 * the fused steps above N_d = 16 and with fp32 slices at 5, 7 and 9..11
 * (where two stages fit), the bucket all-reduce at N_d = 4 and 8 on
 * buckets of at least 32M elements and above N_d = 16 on every bucket, the
 * check above N_d = 16 (with fp32 slices at every N_d but 1, 2, 4 and 8),
 * the accumulation never; the fused DDP step, the fused last micro-batch
 * and the FSDP2 step without the chunk-cat are register-staged only.  The copies (flat_pack, ag_unpack, FSDP2 chunk-cat /
 * copy-out) send the body of every range between its first and last 16-byte
 * boundary of the destination to a 16-byte vector copy (realigning the
 * source when it is not congruent) except under _REGISTER, which keeps them
 * on the generic segment copy.  All give bit-identical results.  Returns the
 * previous setting, or INVALID for an unknown value. */
#define SHARDSTEP_PATH_AUTO 0
#define SHARDSTEP_PATH_REGISTER 1
#define SHARDSTEP_PATH_TMA 2
int32_t shardstep_set_fused_path(int32_t path);

/* Whether kernels are launched as programmatic dependents of the kernel
 * before them in the stream, process-wide.  The first kernel of a call (the
 * fused steps, the accumulation, the step-state kernels, the first copy of
 * a pack or all-gather) may then be scheduled while its predecessor drains,
 * but waits for that predecessor to complete before it touches memory, so
 * only the launch latency overlaps and stream order holds whatever the
 * predecessor is; the second and later kernels of one call (the buckets of
 * ddp_bucket_allreduce_avg, the copy kernels of fsdp_flat_pack,
 * fsdp_ag_unpack, fsdp2_chunk_cat and fsdp2_all_gather_copy_out: disjoint
 * work) start while the previous one drains and wait for it only before
 * they end.  The first bucket of an all-reduce, the non-finite check and
 * the TMA-staged kernels' first launches stay ordinary launches.  1
 * (default) = yes, 0 = ordinary launches everywhere.  Results do not depend
 * on it.  Returns the previous setting. */
int32_t shardstep_set_dependent_launch(int32_t enable);

/* Sets the shared-memory stages of each TMA-staged launch, process-wide:
 * 0 (default) = enough stages for about 128 KB of tiles in flight per SM
 * (at least 2, at most 16); 2..16 = that many, or as many as fit if fewer,
 * rounded down to one of the instantiated counts 2, 3, 4, 6, 8, 12, 16.
 * A tuning control only: results do not depend on it.  Returns the previous
 * setting, or INVALID for other values. */
int32_t shardstep_set_tma_stages(int32_t stages);

/* Watchdog word of the current device: bit 0 = a consumer's wait for a
 * staged tile ran out, bit 1 = the producer's wait for a free stage ran out
 * (in either case the launch returned early and its results are
 * incomplete), bit 2 = the producer's wait for its own copies in flight ran
 * out before the block exited (never expected: those copies read validated
 * device memory).  0 means every TMA-staged launch so far completed its
 * waits.  Synchronous (copies the word to *status); clear != 0 resets it
 * afterwards.  Errors: INVALID (NULL), CUDA. */
int shardstep_device_status(uint32_t* status, int32_t clear);

/* Sets how long a TMA-staged kernel's waits for a staged tile or a free
 * stage may last before the kernel gives up (status bits 0 and 1), in ns,
 * process-wide, read at each launch: 0 = the default of about two seconds.
 * A control for tests that make a wait run out: limits below 1 ms poll
 * without blocking and read the clock after every poll (slower, but such a
 * wait runs out even when each blocking poll would have lasted until its
 * copy landed).  The wait of a block for its own bulk copies before it
 * exits keeps its fixed two-second limit, so no setting lets a block exit
 * with a copy in flight.  Returns the previous limit, or INVALID for
 * ns < 0. */
int64_t shardstep_set_tma_wait_ns(int64_t ns);

/* shardstep_check_mean_division -- device, one launch (self-check).
 * Every reduce here ends with a division by N_d ([P3] section 2: the mean of
 * the N_d local-mean gradients), computed without a divide instruction when
 * N_d is known in advance: a multiply by the exact reciprocal for a power of
 * two, else a multiply by RN(1/N_d) and one fma correction (Markstein).
 * This call runs that division and IEEE fp32 division on all 2^32 fp32 bit
 * patterns and counts the patterns whose results differ in any bit.
 *   nd          1..SHARDSTEP_MAX_ND.
 *   mismatches  device uint64, 8-byte aligned: the count is added to it
 *               (the caller zeroes it first).
 *   first_bad   device uint32: lowered to the smallest differing pattern
 *               (the caller sets it to 0xFFFFFFFF first).
 * Errors: INVALID (nd out of range, NULL, misaligned), CUDA. */
int shardstep_check_mean_division(int32_t nd, uint64_t* mismatches, uint32_t* first_bad,
                                  void* stream);

/* Description of the last error on the calling thread ("" if none). */
const char* shardstep_last_error(void);

/* Kernels this library has launched in this process (all threads). */
uint64_t shardstep_launch_count(void);

/* shardstep_comm_counter -- host only, thread-safe.
 * The emulated collectives move no bytes between GPUs; this counter adds
 * up, over the calls accepted in this process, the bytes their ranks would
 * send if each collective ran as a ring, the model of [P1] ZeRO section and
 * [P3] sections 5 and 8, with the (N_d - 1) / N_d factor kept.  Per call,
 * summed over the shard positions it covers (es = bytes per element of the
 * contributions the kernel reduces: 2 for bf16 / fp16, 4 for fp32 and for
 * the fused last micro-batch, whose contributions are fp32 sums):
 *   a fused step's reduce-scatter   (N_d - 1) * S * es; under hybrid
 *                                   sharding (F - 1) * S * es inside the
 *                                   group + 2 (R - 1) / R * S * es across
 *                                   the R = N_d / F groups;
 *   fsdp_ag_unpack                  (N_d - 1) * S * 2;
 *   fsdp2_all_gather_copy_out       (N_d - 1) * local * es;
 *   a bucket all-reduce (alone or   2 (N_d - 1) / N_d * 2 bytes per bucketed
 *   fused with AdamW)               element;
 *   fsdp_grad_unscale_check         2 (N_d - 1) / N_d * 4 (the found-inf
 *                                   flags OR-ed over the ranks; the reduce
 *                                   is the scaled step's).
 * Packing, accumulation, chunk-cat, views and empty calls count 0.  One rank
 * step of ZeRO-1/2 (a fused step over the rank's shard of every unit, then
 * the all-gather of every unit) thus adds 4 (N_d - 1) / N_d * Psi bytes for
 * Psi padded parameters, and a DDP step 4 (N_d - 1) / N_d * Psi.
 * Returns the running total in bytes; reset != 0 sets it to 0 after reading. */
double shardstep_comm_counter(int32_t reset);

/* Name of the kernel that the calling thread's last successful streaming
 * call launched (fused steps, accumulation, non-finite check; for the bucket
 * all-reduce, the kernel of its last non-empty bucket), e.g.
 * "rs_adamw_cast_vec4<8, bf16> (register-staged)"; "" before the first.
 * Host only; the string stays valid until the thread's next such call. */
const char* shardstep_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* SHARDSTEP_H */
