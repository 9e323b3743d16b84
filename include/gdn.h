/*
 * gdn.h -- C ABI of libgdn: the chunk-parallel (WY form) forward pass of the
 * gated delta rule, GDN and KDA, for NVIDIA GB300 (sm_103a).
 *
 * The operation (stratat pull #1296, "What this is": the gated-delta-net
 * recurrence rewritten in the chunk-parallel WY form; ROCm/rocm-libraries
 * PR #11223, "Summary": KDA prefill with six state-independent tiles plus a
 * serial state recurrence).  For every sequence and value head hv, with the
 * fp32 state S (dk x dv, K-first: row = key channel, logismos issue #46
 * "Verified implementation boundary") and t = 1..L:
 *
 *     S_t = diag(a_t) S_{t-1} + beta_t k_t (v_t - (diag(a_t) S_{t-1})^T k_t)^T
 *     o_t = scale * S_t^T q_t
 *
 * with a_t = exp(g_t): natural-log decay (issue #46, Sep 8 comment), one
 * scalar per (token, value head) for GDN, one per key channel for KDA.  The
 * value head hv reads q/k head hv / (HV / H) (grouped heads, same comment).
 * The input state h0 is never written; the final state goes to a separate
 * buffer hT (issue #46: immutable input state, separate output/next-state).
 *
 * Inside, the work is split in two kernels launched back to back on the
 * caller's stream: a state-independent chunk-prep kernel, parallel over all
 * (chunk, value head), and a scan kernel, serial over the chunks of each
 * sequence and parallel over (sequence, value head, dv slice) (the split
 * composition of PR #11223, "Summary").  The prep kernel's tiles cross to the
 * scan kernel through the caller's workspace.
 *
 * Conventions common to every entry point
 *  - Every pointer argument except `flags_out` is a DEVICE pointer.
 *  - Ownership: the caller allocates every buffer, workspace included; the
 *    library allocates no memory, keeps no per-call state and may be called
 *    from several host threads at once.  The one-time lookup of the driver's
 *    tensor-map encoder is guarded internally; a kernel's shared-memory size
 *    attribute is set at each launch, which the CUDA runtime makes safe from
 *    several threads.
 *  - Asynchrony: work is enqueued on `stream` (NULL = legacy default stream)
 *    and the call returns without synchronising.  Errors of the launch itself
 *    are returned as GDN_ERR_CUDA; faults during execution surface at the
 *    caller's next synchronisation.
 *  - Errors: all argument checks run before anything is enqueued; a call that
 *    returns anything but GDN_OK has enqueued nothing and written nothing.
 *    Nothing aborts, throws or prints across the ABI.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that callers need no CUDA
 * headers. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, aliasing */
  GDN_ERR_UNSUPPORTED = 2, /* a valid request outside the compiled domain */
  GDN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  GDN_ERR_CUDA = 4         /* the CUDA runtime refused a launch or attribute */
} gdn_status;

typedef enum gdn_gate_mode {
  GDN_GATE_SCALAR = 0,  /* GDN: g is [.., HV], one log-gate per value head */
  GDN_GATE_PER_KEY = 1  /* KDA: g is [.., HV, dk], one per key channel */
} gdn_gate_mode;

typedef enum gdn_dtype {
  GDN_F32 = 0,  /* q, k, v, o are float32 */
  GDN_BF16 = 1  /* q, k, v, o are bfloat16 */
} gdn_dtype;

typedef enum gdn_activation {
  GDN_ACT_NONE = 0,  /* identity */
  GDN_ACT_SILU = 1   /* x * sigmoid(x) */
} gdn_activation;

/* Bits of the device status word kept in the first bytes of the workspace. */
enum {
  GDN_FLAG_POSITIVE_GATE = 1u << 0, /* some log-gate g > 0 (a decay above 1) */
  GDN_FLAG_NONFINITE = 1u << 1,     /* a non-finite value was written to o/hT */
  GDN_FLAG_BAD_SEQLENS = 1u << 2,   /* cu_seqlens not 0 = c0 <= c1 <= .. = T;
                                       affected sequences were skipped */
  GDN_FLAG_TIMEOUT = 1u << 3,       /* an internal wait ran out of its time
                                       budget; the results are not valid */
  GDN_FLAG_LAUNCH_CONFIG = 1u << 4  /* a kernel received dynamic shared memory
                                       without the alignment its operand
                                       images need and did no work; the
                                       results are not valid */
};

/* Library version, major*10000 + minor*100 + patch. */
GDN_API int gdn_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
GDN_API const char *gdn_status_string(int status);

/*
 * Bytes of workspace gdn_chunk_fwd needs for this problem; 0 for a request
 * that gdn_chunk_fwd would reject.  Arguments as for gdn_chunk_fwd
 * (n_seqs = number of packed sequences when cu_seqlens is used, else B).
 * The value does not depend on the contents of cu_seqlens.
 */
GDN_API size_t gdn_chunk_fwd_workspace_bytes(int B, int T, int H, int HV, int dk,
                                     int dv, int chunk, int gate_mode,
                                     int n_seqs, int dtype);

/*
 * Forward pass of the gated delta rule in chunk-parallel WY form.
 *
 * Layouts (contiguous, row-major; "dt" = dtype):
 *   q, k   [B, T, H, dk]   dt          v, o   [B, T, HV, dv]   dt
 *   g      [B, T, HV] (GDN) or [B, T, HV, dk] (KDA)          fp32, <= 0
 *   beta   [B, T, HV]                                          fp32
 *   h0, hT [N, HV, dk, dv]  fp32, K-first (N = B, or n_seqs when packed)
 *   cu_seqlens  [n_seqs + 1] int32, device; packed sequences (then B == 1
 *               and T is the total token count); NULL for plain batches.
 *
 * h0 may be NULL (zero initial state); hT may be NULL (final state not
 * written).  hT must not overlap h0, and o must not overlap q, k, v, g or
 * beta.  Every pointer must be 16-byte aligned.  scale multiplies the read
 * (dk^-0.5 is usual).  chunk is the sub-chunk length C of the WY form.
 *
 * Supported domain: dk, dv in {64, 128}; chunk in {32, 64}; dtype F32 or BF16;
 * HV a multiple of H.  Anything else valid returns GDN_ERR_UNSUPPORTED.
 * Packed sequences of length 0 are allowed: their hT is h0 (or 0).
 * T == 0 is allowed; q, k, v, g, beta and o may then be NULL.
 *
 * Workspace: at least gdn_chunk_fwd_workspace_bytes(...) bytes, 256-byte
 * aligned, owned by the caller, not shared by two calls in flight.  Its first
 * 256 bytes hold the device status word (GDN_FLAG_*), cleared by each call;
 * read it back with gdn_read_device_flags.
 *
 * Numerics: fp32 state, fp32 accumulation, o rounded once to dtype.  fp32
 * inputs: every product keeps at least 16 mantissa bits (operands split into
 * two bf16 halves).  bf16 inputs: tensor-core operands are fp16 (11 mantissa
 * bits; key, query, state and per-chunk tiles must stay below 65504 in
 * magnitude, which unit-norm keys/queries and decays <= 1 guarantee), and the
 * per-chunk solve runs in fp32.
 */
GDN_API gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *g, const float *beta, const float *h0,
                         void *o, float *hT, const int32_t *cu_seqlens,
                         int n_seqs, int B, int T, int H, int HV, int dk,
                         int dv, int chunk, float scale, int gate_mode,
                         int dtype, void *workspace, size_t workspace_bytes,
                         gdn_stream_t stream);

/*
 * The two halves of gdn_chunk_fwd, for callers that schedule them apart (to
 * time each kernel, or to overlap one layer's prep with another's scan).
 * Same arguments and checks as gdn_chunk_fwd.  gdn_chunk_fwd_prep clears the
 * status word and runs the state-independent chunk-prep kernel, which writes
 * the per-chunk tiles into `workspace` (it reads q, k, g, beta, cu_seqlens);
 * gdn_chunk_fwd_scan runs the serial scan kernel, which reads those tiles and
 * writes o and hT.  A scan must follow, in stream order, a prep with the same
 * arguments and workspace; gdn_chunk_fwd_prep followed by gdn_chunk_fwd_scan
 * computes exactly what gdn_chunk_fwd computes.
 */
/*
 * gdn_chunk_fwd with its two kernels in one launch, in lockstep: the fused
 * prep + scan composition of ROCm/rocm-libraries PR #11223 ("Summary"), built
 * for this GPU as a cooperative grid.  Its first CTAs run the scan's blocks;
 * the rest run the chunk prep in persistent warpgroups, chunk by chunk, and
 * set a ready flag per (chunk, q/k head) in the workspace once that unit's
 * operand images are complete; the scan loads an image only after its flag
 * (bounded wait: GDN_FLAG_TIMEOUT if a flag never comes).  Same arguments,
 * checks, workspace and results as gdn_chunk_fwd, bit for bit: both run the
 * same per-chunk and per-block device code.  Only the bf16 scalar-gate (GDN)
 * path has it: other dtype / gate combinations return GDN_ERR_UNSUPPORTED,
 * as does a problem whose scan blocks (sequences x HV x dv/64) leave no SM
 * for the prep.  The prep gets a head start: the split prep kernel covers the
 * first chunk slots on every SM (half of them at 32k tokens, more for shorter
 * inputs: enough that the prep warpgroups can finish the rest while the scan
 * walks its chunks), enqueued just before the cooperative launch.  A call that
 * must finish before the next work starts is faster this way from about 8192
 * tokens up (measured: 0.87 ms against 1.01 ms for gdn_chunk_fwd on 32k
 * tokens, 16 q/k and 48 value heads of 128; at 2048 and 4096 tokens the two
 * are within 3%); independent calls in flight on several streams are faster
 * with gdn_chunk_fwd, whose kernels can share the GPU, while cooperative
 * launches run one at a time (PR #11223, "Notes for reviewers": the
 * composition is chosen by measurement).
 */
GDN_API gdn_status gdn_chunk_fwd_lockstep(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, const float *h0,
                              void *o, float *hT, const int32_t *cu_seqlens,
                              int n_seqs, int B, int T, int H, int HV, int dk,
                              int dv, int chunk, float scale, int gate_mode,
                              int dtype, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream);

GDN_API gdn_status gdn_chunk_fwd_prep(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, const float *h0,
                              void *o, float *hT, const int32_t *cu_seqlens,
                              int n_seqs, int B, int T, int H, int HV, int dk,
                              int dv, int chunk, float scale, int gate_mode,
                              int dtype, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream);
GDN_API gdn_status gdn_chunk_fwd_scan(const void *q, const void *k, const void *v,
                              const float *g, const float *beta, const float *h0,
                              void *o, float *hT, const int32_t *cu_seqlens,
                              int n_seqs, int B, int T, int H, int HV, int dk,
                              int dv, int chunk, float scale, int gate_mode,
                              int dtype, void *workspace, size_t workspace_bytes,
                              gdn_stream_t stream);

/*
 * gdn_chunk_fwd for callers that cannot allocate device memory: a component
 * inside a host framework that owns all device memory and gives it no
 * allocation of its own, or a latency-critical loop that must not stall on
 * an allocation.  (The pages describe no such entry point; it has no
 * counterpart there.)
 *
 * Same arguments, layouts, checks and results as gdn_chunk_fwd, minus the
 * workspace: the library uses a fixed 64 MiB device array of its own instead,
 * reserved on every GPU that loads the library until the process exits.  The
 * caller still provides q, k, v, g, beta, h0, o and hT.  Returns
 * GDN_ERR_WORKSPACE when the request needs more than 64 MiB of workspace
 * (gdn_chunk_fwd_workspace_bytes tells), GDN_ERR_CUDA when the array's
 * device address cannot be obtained.  The first call on each device looks
 * that address up (with the device current); make that first call before any
 * stream capture.  All calls on a device share the one array: calls that
 * overlap on the GPU race and must be serialised by the caller.  The device
 * status word of these calls lives in that array and is not exposed, so what
 * the kernels find on the device (a wait that ran out, malformed cu_seqlens,
 * a non-finite result, a positive log-gate) cannot be detected through this
 * entry point: the call still returns GDN_OK.  A caller that needs that
 * status uses gdn_chunk_fwd with a workspace of its own and reads it with
 * gdn_read_device_flags.
 */
GDN_API gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta,
                                 const float *h0, void *o, float *hT,
                                 const int32_t *cu_seqlens, int n_seqs, int B,
                                 int T, int H, int HV, int dk, int dv, int chunk,
                                 float scale, int gate_mode, int dtype,
                                 gdn_stream_t stream);

/*
 * The token-serial (recurrent) form of the same recurrence: each sequence's
 * tokens one after another, the state held on chip between them.  With T == 1
 * this is the decode step (logismos issue #46, "Verified implementation
 * boundary": a one-token grouped step, K-first input state, separate output
 * and next-state buffers, value width up to 1024); with T > 1 it is the
 * plain definition that gdn_chunk_fwd reaches by the chunked route, useful
 * for short prompts and continuation of a few tokens.
 *
 * Arguments, layouts and the grouped-head mapping are those of gdn_chunk_fwd,
 * without chunk and workspace.  Differences:
 *  - dk in {64, 128}; dv any multiple of 32 up to 1024.
 *  - hT may be h0 itself (the same pointer): the state is then updated in
 *    place, as a decode loop over a state cache wants.  Any other overlap of
 *    hT with h0 is refused.
 *  - flags: a DEVICE pointer to one uint32 (4-byte aligned) or NULL.  When
 *    given, the call clears it, then sets GDN_FLAG_* bits as gdn_chunk_fwd
 *    does in its workspace (POSITIVE_GATE, NONFINITE, BAD_SEQLENS);
 *    gdn_read_device_flags(flags, ...) reads it back.
 * No workspace is needed and nothing else is written.
 *
 * Numerics: fp32 state and arithmetic throughout (no tensor-core operands),
 * o rounded once to dtype.
 */
GDN_API gdn_status gdn_recurrent_fwd(const void *q, const void *k, const void *v,
                                     const float *g, const float *beta, const float *h0,
                                     void *o, float *hT, const int32_t *cu_seqlens,
                                     int n_seqs, int B, int T, int H, int HV, int dk,
                                     int dv, float scale, int gate_mode, int dtype,
                                     uint32_t *flags, gdn_stream_t stream);

/*
 * Operations either side of the recurrence.  The pages keep them out of the
 * recurrence's own contract (logismos issue #46, "Remaining work": gating,
 * packing and convolution compose separately from the generic operation), so
 * they are entry points of their own, each one memory-bound kernel.
 *
 * gdn_causal_conv1d_fwd -- causal depthwise convolution over time with a
 * raw-input history (issue #46, "Verified implementation boundary": the
 * staged causal convolution step keeps a channel-major, oldest-to-newest raw
 * history, writes the next history and the output to separate buffers, and
 * has no history for width 1).  For each sequence, channel c and
 * ext = [history of c; x of c]:
 *     y[t, c] = act(bias[c] + sum_{j < W} w[c, j] * ext[t + j])
 * (w[c, W-1] weighs the current input), and the next history is the last
 * W - 1 entries of ext, so a sequence shorter than W - 1 keeps part of the
 * old one.  Layouts: x, y [B, T, D] (or packed [1, Ttot, D] with cu_seqlens)
 * in dtype; w [D, W], bias [D] (or NULL), h0, hT [N, D, W-1] fp32 (h0 NULL =
 * zeros; hT NULL = not written; hT may be h0 itself).  y must not overlap x.
 * Supported: W in 1..4, D a multiple of 8, dtype F32 or BF16, activation
 * GDN_ACT_NONE or GDN_ACT_SILU.  flags: as for gdn_recurrent_fwd
 * (GDN_FLAG_BAD_SEQLENS).  With T == 1 this is the one-token decode step.
 */
GDN_API gdn_status gdn_causal_conv1d_fwd(const void *x, const float *w, const float *bias,
                                         const float *h0, void *y, float *hT,
                                         const int32_t *cu_seqlens, int n_seqs, int B, int T,
                                         int D, int width, int activation, int dtype,
                                         uint32_t *flags, gdn_stream_t stream);

/*
 * gdn_l2norm_fwd -- rows of x ([rows, dim], dtype) divided by
 * sqrt(sum of squares + eps): the unit-norm queries and keys the recurrence
 * expects.  y may be x itself.  dim in {64, 128, 256}.
 */
GDN_API gdn_status gdn_l2norm_fwd(const void *x, void *y, int64_t rows, int dim, float eps,
                                  int dtype, gdn_stream_t stream);

/*
 * gdn_rmsnorm_gated_fwd -- the output norm that follows the recurrence
 * (stratat pull #1296, re-base notes; the pages print no formula, and this is
 * the plain reading): per row of x ([rows, dim], dtype)
 *     y = x / sqrt(mean(x^2) + eps) * weight * silu(z)     (z NULL: no gate)
 * with weight [dim] fp32 and z [rows, dim] in dtype.  y may be x itself.
 * dim in {64, 128, 256}.
 */
GDN_API gdn_status gdn_rmsnorm_gated_fwd(const void *x, const void *z, const float *weight,
                                         void *y, int64_t rows, int dim, float eps, int dtype,
                                         gdn_stream_t stream);

/*
 * gdn_state_combine -- compose a segment's state transfer.  Over any run of a
 * sequence's tokens the recurrence maps its entering state affinely,
 * S_out = M S_in + S_seg, with S_seg the state the run leaves from a zero
 * start (gdn_chunk_fwd with h0 = NULL) and M the state it leaves from the
 * identity with all values zero (gdn_chunk_fwd with v = 0, dv = dk, h0 = I).
 * A sequence split into segments on several GPUs exchanges (M, S_seg) per
 * segment and composes them with this product (the state-transfer exchange
 * for sequences longer than one GPU's share; logismos issue #46, "Remaining
 * work", later continuation).  Per state n < n_seqs and value head:
 *     S_out = M S_in + S_seg,  M [n_seqs, HV, dk, dk], the others
 *     [n_seqs, HV, dk, dv], all fp32, device pointers, 16-byte aligned.
 * S_out may be S_seg itself; it must not overlap M or S_in.  dk, dv <= 1024.
 */
GDN_API gdn_status gdn_state_combine(const float *M, const float *S_in, const float *S_seg,
                                     float *S_out, int n_seqs, int HV, int dk, int dv,
                                     gdn_stream_t stream);

/*
 * gdn_selftest_wait -- exercise the bounded wait that every mbarrier wait of
 * the tensor-core kernels uses, with no fault and no hang.  Those waits give
 * up after a clock budget (about two seconds), set GDN_FLAG_TIMEOUT and let
 * the kernel finish, so that a completion that never comes ends as a status,
 * not a hung GPU.  This call clears the uint32 at `flags` (DEVICE pointer,
 * 4-byte aligned), then runs one 32-thread block that waits, with a budget of
 * `budget_cycles` SM clock cycles (1 .. 4e9), on a barrier of its own:
 * complete = 0: nothing arrives, every wait runs out and *flags becomes
 * GDN_FLAG_TIMEOUT; complete = 1: the barrier completes first and *flags stays
 * 0.  Read the word back with gdn_read_device_flags(flags, ...).
 * (Failure detection the pages ask for in spirit -- invalid work is refused
 * before publication, logismos issue #46; they describe no such entry point.)
 */
GDN_API gdn_status gdn_selftest_wait(uint32_t *flags, long long budget_cycles, int complete,
                                     gdn_stream_t stream);

/*
 * Copy the device status word of `workspace` to *flags_out (host pointer)
 * after all work queued on `stream` so far has finished (synchronises the
 * stream).  Returns GDN_ERR_INVALID_ARG for NULL arguments and GDN_ERR_CUDA
 * if the copy fails (including an earlier asynchronous fault).
 */
GDN_API gdn_status gdn_read_device_flags(const void *workspace, uint32_t *flags_out,
                                 gdn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
