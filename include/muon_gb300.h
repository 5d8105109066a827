/*
 * muon_gb300.h -- C ABI of the GB300 (sm_103a) Muon optimizer step.
 *
 * The Muon step, as the pages describe it:
 *   [MCS] "Muon Custom Sizing 实战：modded-nanogpt 将注意力与 MLP 参数合并进同一
 *         reduce_scatter 调用，把 124M GPT 训练压进 150 秒", section 2.3 (batched
 *         NS of the QKVO view, coefficients (a,b,c) = (3.4445, -4.7750, 2.0315),
 *         five rounds) and section 四 (momentum lerp, Nesterov blend, decoupled
 *         decay lr*wd, write-back with alpha = -lr * max(1, hdim/dim)^0.5);
 *   [PG]  "parameter-golf train_gpt.py 源码精读：Muon 优化器、Int8 量化与 DDP 数据
 *         加载全解", part 1, section 核心思想 (the Newton-Schulz function:
 *         X /= ||X||; repeat A = X X^T, B = bA + cA^2, X = aX + BX) and section
 *         分布式细节 (rescale of the result by max(1, m/n)^0.5).
 *
 * Conventions shared by every entry point:
 *   - Matrices are row-major and contiguous, stacked as [batch, rows, cols].
 *     A stack of same-shape weights is one call; the [MCS] QKVO weight stored
 *     as (hdim, 4*dim) is passed as batch 4 of (hdim, dim): the same bytes.
 *   - Every data pointer is device memory owned by the caller, 16-byte
 *     aligned.  Parameters and momentum buffers are updated in place;
 *     gradients are only read.  No call allocates device memory; the one
 *     device memory the library itself holds is the fixed 64 MiB scratch of
 *     muon_step_noalloc(), a static array that every GPU which loads the
 *     library keeps until the process exits.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     work is enqueued on it asynchronously; no entry point synchronises
 *     except muon_workspace_status().
 *   - The workspace is caller-owned device memory of at least the size that
 *     muon_workspace_bytes()/muon_grouped_workspace_bytes() return, 256-byte
 *     aligned, and zero-filled before its first use (it carries a sticky
 *     device error word).  Calls that share a workspace must not overlap on
 *     the GPU.
 *   - Failure (no counterpart on the pages): every device-side wait is
 *     bounded (2 s).  A wait that gives up sets the workspace's error word;
 *     from then on the waits of the other kernels still running end within
 *     microseconds, and every kernel of every later call on that workspace
 *     returns at entry, so those calls change nothing (parameters, momentum
 *     and outputs keep their values) until muon_workspace_status() clears
 *     the word.  The call during which the wait gave up may have written part
 *     of its results.
 *   - Argument errors are reported before anything is enqueued.  A CUDA error
 *     while enqueuing gives MUON_ERR_CUDA.  No C++ exception crosses the ABI.
 *   - NS runs in bf16 on the tensor cores (fp32 accumulation and epilogues)
 *     for min(rows, cols) >= 64; smaller matrices run the same iteration in
 *     fp32 on the CUDA cores (bf16 is too coarse for, e.g., a 1x12 gate).
 *   - When rows > cols the iteration runs on the transpose (A is the
 *     min(rows,cols)^2 Gram matrix); the result comes back in the input's
 *     orientation.  The norm is Frobenius, divided as ||X||_F + eps.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum muon_status {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment, dtype or scalar     */
  MUON_ERR_UNSUPPORTED = 2,  /* no sm_103a device current, or shape out of range  */
  MUON_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed                 */
  MUON_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up (see status)   */
  MUON_ERR_WORKSPACE = 5     /* workspace NULL, misaligned or too small           */
} muon_status;

typedef enum muon_dtype {
  MUON_F32 = 0,
  MUON_BF16 = 1
} muon_dtype;

/* One stack of same-shape 2-D weights for muon_step_grouped(). */
typedef struct muon_group {
  float* params;        /* [batch, rows, cols] fp32, updated in place            */
  const void* grads;    /* [batch, rows, cols] in g_dtype, read only             */
  float* momentum_buf;  /* [batch, rows, cols] fp32, updated in place            */
  int g_dtype;          /* muon_dtype of grads                                   */
  int batch;            /* 0..65535; 0 skips the group                           */
  int rows, cols;       /* >= 1 each, <= 65536 each                              */
  float lr_scale;       /* <= 0: max(1, rows/cols)^0.5 ([PG] 分布式细节)          */
} muon_group;

/* Kinds of kernel the library launches (trace records, launch counts). */
typedef enum muon_kernel_kind {
  MUON_K_PROLOGUE = 0,   /* momentum, Nesterov blend, bf16 cast, norm partials  */
  MUON_K_SMALL_NS = 1,   /* whole step in fp32 for min(rows,cols) < 64          */
  MUON_K_GRAM = 2,       /* A = s^2 X X^T, upper 256 x 256 tiles only           */
  MUON_K_POLY = 3,       /* B' = a I + b A + c A A, upper 256 x 256 tiles only  */
  MUON_K_UPDATE = 4,     /* X <- s B' X  (= s (a X + B X))                      */
  MUON_K_APPLY = 5,      /* p <- (1 - lr wd) p - lr scale O (or O as bf16)      */
  MUON_K_ADAM = 6,       /* DistAdam update of non-matrix parameters            */
  MUON_K_FUSED_NS = 7,   /* all NS rounds, one CTA pair per matrix, 64<=m<=256,
                            n<=512 (see muon_set_fused_ns)                      */
  MUON_K_ROUNDS = 8      /* all Gram/Poly/Update stages of every round in one
                            persistent launch (see muon_set_persistent_rounds)  */
} muon_kernel_kind;

/* Workspace bytes for one muon_step()/muon_ns5() call on [batch, rows, cols].
 * Returns 0 if the sizes are invalid. */
size_t muon_workspace_bytes(int batch, int rows, int cols);

/* Workspace bytes for one muon_step_grouped() call; 0 if a group is invalid. */
size_t muon_grouped_workspace_bytes(const muon_group* groups, int n_groups);

/*
 * The Newton-Schulz function ([PG] 核心思想) on every matrix of a stack:
 *   X = G / (||G||_F + eps)  (on G^T if rows > cols),
 *   `steps` times: A = X X^T;  B = b A + c A A;  X = a X + B X,
 *   out = X (transposed back), written as bf16 [batch, rows, cols].
 * G: [batch, rows, cols] fp32 or bf16 (g_dtype).  steps in 1..16; batch in
 * 0..65535, rows and cols in 1..65536 (the same limits hold for every call).
 */
muon_status muon_ns5(const void* G, int g_dtype, void* out_bf16,
                     int batch, int rows, int cols, int steps,
                     float a, float b, float c, float eps,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * One Muon step on a stack of same-shape weights ([MCS] 四, [PG] 核心思想/分布式细节):
 *   buf <- buf + (1 - momentum) (g - buf)
 *   u   <- g + momentum (buf - g)  if nesterov, else buf
 *   O   <- NS(u) as in muon_ns5 (bf16, as the last Newton-Schulz update writes it)
 *   p   <- (1 - lr weight_decay) p - lr s O,   s = lr_scale > 0 ? lr_scale
 *                                                 : max(1, rows/cols)^0.5
 * momentum in [0, 1]; steps in 1..16; eps >= 0; all scalars finite.
 */
muon_status muon_step(float* params, const void* grads, int g_dtype, float* momentum_buf,
                      int batch, int rows, int cols,
                      float momentum, int nesterov, float lr, float weight_decay,
                      float lr_scale, int steps, float a, float b, float c, float eps,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * muon_step without a workspace, for callers that cannot call cudaMalloc: code
 * running under an allocator that has already reserved the whole GPU, plug-ins
 * allowed to touch only the memory they are handed, or training loops that
 * forbid any allocation after start-up.  The pages have no counterpart: this is
 * an interface addition, not part of the method.
 * Arguments and results are those of muon_step, minus the workspace.  Scratch is
 * a 64 MiB array built into the library (held by every GPU that loads it until
 * the process exits); a call whose muon_workspace_bytes(batch, rows, cols)
 * exceeds 64 MiB returns MUON_ERR_WORKSPACE.  The first call on a device looks
 * up the array's device address, so make it before any stream capture.  All
 * calls on a device share the array: calls that overlap on the GPU race.
 * Each call clears the array's sticky error word on `stream` after its
 * argument checks and before its first kernel, so the word reports the latest
 * call on the device: read it with muon_noalloc_status().
 */
muon_status muon_step_noalloc(float* params, const void* grads, int g_dtype, float* momentum_buf,
                              int batch, int rows, int cols,
                              float momentum, int nesterov, float lr, float weight_decay,
                              float lr_scale, int steps, float a, float b, float c, float eps,
                              void* stream);

/*
 * muon_workspace_status() for the built-in scratch of muon_step_noalloc() on
 * the current device (no counterpart on the pages): synchronises `stream`,
 * then returns MUON_OK, or MUON_ERR_TIMEOUT if a bounded device-side wait
 * gave up during the latest muon_step_noalloc() call on this device (or
 * during a muon_selftest_wait_timeout() on the scratch since).  clear != 0
 * resets the word afterwards.
 */
muon_status muon_noalloc_status(void* stream, int clear);

/*
 * muon_step on every group of a model at once (the pages stack the weights of
 * each parameter group, [MCS] 四 第一遍/第二遍).  Groups share the scalars; the
 * NS rounds of all tensor-core groups run as one grouped launch per stage.
 * n_groups >= 0; groups may be NULL only when n_groups == 0.  The arrays of
 * different groups must not overlap.
 */
muon_status muon_step_grouped(const muon_group* groups, int n_groups,
                              float momentum, int nesterov, float lr, float weight_decay,
                              int steps, float a, float b, float c, float eps,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads the workspace's sticky device error word:
 * MUON_OK, or MUON_ERR_TIMEOUT if a bounded wait inside a kernel gave up since
 * the word was last cleared.  clear != 0 resets the word to zero afterwards.
 */
muon_status muon_workspace_status(const void* workspace, size_t workspace_bytes,
                                  void* stream, int clear);

/*
 * Self-test of the device-side timeout path (no counterpart on the pages).
 * Enqueues one kernel whose bounded wait, the same code every GEMM role waits
 * with, is on a barrier that nothing completes; after `limit_us` (1..100000)
 * it gives up and records the timeout in the workspace's status word, as a
 * stalled GEMM would.  muon_workspace_status() then reports MUON_ERR_TIMEOUT.
 * workspace = NULL targets the built-in scratch of muon_step_noalloc() on the
 * current device instead (workspace_bytes is then ignored), read back with
 * muon_noalloc_status().  Nothing faults, hangs or is left pending on the GPU.
 */
muon_status muon_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int limit_us,
                                       void* stream);

/*
 * The Adam half of the optimizer: the DistAdam update that trains the
 * parameters Muon does not take (embeddings, output head, {0,1}-D scalars).
 * Defined by the DistAdam step() printed in "将 Adam 梯度同步（Reduce-Scatter）
 * 移入反向 Hook：modded-nanogpt 分布式优化器每步提速约 0.7 秒的工程实践",
 * section 改动二, with lr_eff = lr * lr_scale and t = `step`:
 *   if weight_decay != 0:  p *= 1 - lr_eff * weight_decay * wd_scale
 *   m = beta1 m + (1 - beta1) g;   v = beta2 v + (1 - beta2) g^2
 *   p -= lr_eff * sqrt(1 - beta2^t) / (1 - beta1^t) * m / (sqrt(v) + eps)
 * ([MCS] section 四 gives lr 0.008, betas (0.8, 0.95), eps 1e-8 for it.)
 * On one GPU the reduce-scatter / all-gather of that page has no work: each
 * tensor is updated whole, as one flat array of `numel` elements.
 */
typedef struct muon_adam_tensor {
  float* param;         /* [numel] fp32, updated in place                        */
  const void* grad;     /* [numel] in g_dtype, read only                         */
  float* exp_avg;       /* [numel] fp32 first moment m, updated in place         */
  float* exp_avg_sq;    /* [numel] fp32 second moment v, updated in place        */
  long long numel;      /* >= 0; 0 skips the tensor (its pointers may be NULL)   */
  int g_dtype;          /* muon_dtype of grad                                    */
  float lr_scale;       /* per-parameter lr multiplier (1 = none), finite, >= 0  */
  float wd_scale;       /* per-parameter weight-decay multiplier (1 = none)      */
} muon_adam_tensor;

/*
 * One Adam step over n_tensors >= 0 tensors (tensors may be NULL only when
 * n_tensors == 0), all at step count `step` >= 1 (the value after the
 * increment).  0 <= beta1, beta2 < 1; eps >= 0; lr and weight_decay finite.
 * Pointers 16-byte aligned; the arrays of different tensors must not overlap.
 * Up to 64 tensors go in one kernel launch; more take one launch per 64.
 * Needs no workspace and has no waits.
 */
muon_status muon_adam_step(const muon_adam_tensor* tensors, int n_tensors, int step, float lr,
                           float beta1, float beta2, float eps, float weight_decay,
                           void* stream);

/*
 * Path selection (no counterpart on the pages).  With enable = 1 (the default)
 * every matrix with 64 <= min(rows, cols) <= 256 and max(rows, cols) <= 512
 * runs all its NS rounds in one kernel, one CTA pair per matrix, with X, A and
 * B' held on chip between rounds; enable = 0 sends it through the staged
 * tensor-core path (three GEMM launches per round, with A and B' in the
 * workspace).  The grouped prologue and apply are the same on both paths.
 * A call that also holds matrices outside that range (which need the staged
 * launches) runs all of them staged, since the fused kernel would run before
 * the staged chain rather than beside it.
 * Both compute the same step and need the same workspace size.  Process-wide;
 * affects calls made afterwards.  Returns the previous setting, or -1 (nothing
 * changed) if enable is not 0 or 1.
 */
int muon_set_fused_ns(int enable);

/*
 * Launch structure of the tensor-core NS rounds (no counterpart on the pages).
 * mode = 0: one grouped launch per stage and round (Gram, Poly, Update; 15
 * launches for five rounds), each waiting for the one before.
 * mode = 1: one persistent launch covers every stage of every round; a tile
 * starts as soon as the tiles of the stages before it of the same matrix are
 * stored (per-matrix completion counters in the workspace), so one matrix's
 * next stage overlaps other matrices' current one.
 * mode = 2 (the default): 1 for groups whose rounds are short (estimated
 * tensor-core time of a round under 400 us), where the stage boundaries weigh
 * most; 0 otherwise.  Same results and workspace size in every mode.
 * The persistent launch needs all of its clusters (one per two SMs that fit
 * at once) resident together, since tiles wait for tiles of other clusters:
 * kernels on other streams that hold SMs delay it, and if they hold them for
 * more than its 2 s wait limit the step reports MUON_ERR_TIMEOUT.  Mode 0 has
 * no such requirement.
 * Process-wide; affects calls made afterwards.  Returns the previous mode, or
 * -1 (nothing changed) if mode is not 0, 1 or 2.
 */
int muon_set_persistent_rounds(int mode);

/*
 * Where the parameter write runs (no counterpart on the pages).  enable = 1
 * (the default): when every tensor-core matrix of a muon_step or
 * muon_step_grouped call goes through one staged NS chain (one persistent
 * rounds launch, or one launch per stage and round; see above), every weight's
 * cols is a multiple of 8, and rows and cols of every rows > cols weight are
 * multiples of 8, the write is launched right behind the last update (the
 * rounds kernel, or the last round's update launch) and runs beside it: its
 * blocks take the matrices in the order that update ends them (waiting,
 * bounded, on per-matrix completion counters), and the last round stores O of
 * a rows > cols matrix already transposed.  enable = 0: the write runs after
 * the NS.  Same results and workspace size either way; muon_ns5 always uses
 * the second form.
 * Process-wide; affects calls made afterwards.  Returns the previous setting.
 */
int muon_set_streamed_apply(int enable);

/* Static English text for a status code. */
const char* muon_status_string(muon_status status);

/* Kernels this library has launched in this process (all devices, all calls). */
unsigned long long muon_kernel_launch_count(void);

/*
 * Optional kernel timing trace (off by default; host-side bookkeeping only).
 * muon_trace_begin(n): from now on, record a CUDA event before and after each
 * kernel the library launches, on that launch's stream, for up to n launches.
 * muon_trace_end(out, max, &count): synchronise on the recorded events, fill
 * up to `max` records (in launch order), set `count`, and stop tracing.
 * flops/bytes are the launch's algorithmic work: for GEMM stages the dense
 * flops of the tiles the stage is defined on (2 m^2 n for the Gram and for the
 * update, 2 m^3 for the polynomial, each counted once for symmetric outputs
 * as m(m+1)/2 entries), for the prologue the bytes it must move.
 */
typedef struct muon_trace_record {
  int kind;        /* muon_kernel_kind                          */
  int round;       /* NS round (0-based), -1 if not an NS stage */
  float ms;        /* event-to-event time on the launch stream  */
  double flops;    /* algorithmic flops of the launch           */
  double bytes;    /* algorithmic HBM bytes of the launch       */
} muon_trace_record;

muon_status muon_trace_begin(int max_launches);
muon_status muon_trace_end(muon_trace_record* out, int max_records, int* count);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
