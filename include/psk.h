/* psk.h -- C ABI of the fusion-group hot path on one GB300 (sm_103a).
 *
 * Four entry points run the cases of a fusion group on the caller's CUDA
 * stream:
 *
 *   psk_group_run       a connected chain of up to 64 elementwise nodes sharing
 *                       one loop nest, with broadcast inputs
 *                       (PSK-Realize, "What a group is");
 *   psk_softmax_region  the reduction-rooted row region Reduce(Max) -> Sub ->
 *                       Exp -> Reduce(Sum) -> Div with a declared summation
 *                       order (poot "Fusion and Planning", Reduction-rooted
 *                       regions; presk "Native execution", the realization's
 *                       order);
 *   psk_norm_region     the RMSNorm and LayerNorm row regions, the same
 *                       skeleton with their own reductions and epilogues;
 *   psk_adamw_tree      the AdamW step as one parameter-tree group over every
 *                       leaf of a model, in one launch (PSK-Realize, Parameter
 *                       trees; presk "The language", The optimizer).
 *
 * Conventions for every call:
 * - Pointers named ptr/x/y/theta/m/v/grad/gamma/beta/workspace are DEVICE
 *   pointers owned by the caller; descriptor structs and arrays of them are
 *   HOST memory, read during the call only.  The library allocates no device memory and keeps no state
 *   across calls besides cached device attributes and one device status word
 *   (psk_device_status).
 * - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *   stream).  Return 0 means the work was enqueued.
 * - A negative return is a refusal: nothing was launched, and
 *   psk_last_error() (thread-local) names the argument, node or leaf at fault.
 *   Malformed input is refused, never ignored or silently repaired.
 * - Arithmetic is IEEE binary32 with no contraction: every node of a group is
 *   rounded once to f32 and only the root is rounded to its storage type; exp
 *   and erf nodes are correctly rounded.  bf16 is storage only: a shift on
 *   the way in, one round to nearest even on the way out.
 */
#ifndef PSK_H
#define PSK_H

#if !defined(__CUDACC_RTC__)
#include <stdint.h>
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ errors */
#define PSK_OK 0
#define PSK_E_PROGRAM (-1)        /* malformed node program */
#define PSK_E_TOO_MANY_NODES (-2) /* more than 64 op nodes: not one group */
#define PSK_E_SHAPE (-3)          /* shape, stride or size out of range */
#define PSK_E_DTYPE (-4)          /* unknown storage type */
#define PSK_E_NULL (-5)           /* a required pointer is NULL */
#define PSK_E_ORDER (-6)          /* unknown summation order or parameter */
#define PSK_E_CUDA (-7)           /* the CUDA runtime refused the launch */
#define PSK_E_ALIAS (-8)          /* output overlaps an input in a way that races */
#define PSK_E_ARG (-9)            /* any other argument out of range */

/* ------------------------------------------------------- storage types */
/* PSK_I32 (32-bit integers) is a fusion group's input type for SELECT
 * conditions only; every other argument of every entry point refuses it. */
typedef enum { PSK_F32 = 0, PSK_BF16 = 1, PSK_I32 = 2 } psk_dtype;

/* ======================================================== psk_group_run
 * Program format (postfix; one uint32 token per item; opcode in bits 31..24,
 * argument in bits 23..0).  Operand tokens push a value, op tokens pop their
 * operands and push a node (a binary op pops b then a and computes a OP b):
 *   IN k   input k            IMM k  immediate k         REF k  op node k's value
 *   ADD SUB MUL DIV           IEEE binary32, one rounding each
 *   MAX MIN                   max(a,b) = a > b ? a : b, min(a,b) = a < b ? a : b
 *                             (a tie, and NaN, give the second operand)
 *   NEG ABS                   sign flip / sign clear
 *   EXP ERF                   correctly rounded exp / erf
 *   EXPC                      exp(min(max(a, -4), 4))
 *   GELU                      a * (0.5 * (1 + erf(a * RN(1/sqrt 2))))
 *   SQRT SQRTA                sqrt(a) / sqrt(|a|), IEEE
 *   RECIP                     1 / a, IEEE (one rounding)
 *   LOG TANH                  correctly rounded natural log / tanh
 *   SELECT                    c a b SELECT -> a where c != 0, else b; pops b,
 *                             then a, then c.  The condition c must be an IN
 *                             token of a PSK_I32 input, and a PSK_I32 input is
 *                             read only as a condition (else PSK_E_DTYPE at
 *                             run).  The picked value's bits are moved, never
 *                             computed on: a NaN or an infinity in the other
 *                             branch never reaches the result (poot "Fusion
 *                             and Planning", Pointwise chains: Select is a
 *                             bit-moving select on an I32 region input).
 * The op set follows the same passage's unaries (Neg, Exp, Log, Sqrt, Recip,
 * Tanh, Erf) and Select; sigmoid is the chain 1 / (1 + exp(-a)).
 * A valid program has 1..64 op nodes (the cap at which a group stops
 * growing, PSK-Realize "What a group is"), at most 1024 tokens, REFs only to
 * nodes already computed, operands in range, and leaves exactly one value (the
 * root) on the stack. */
#define PSK_OP_IN 0x01
#define PSK_OP_IMM 0x02
#define PSK_OP_REF 0x03
#define PSK_OP_ADD 0x10
#define PSK_OP_SUB 0x11
#define PSK_OP_MUL 0x12
#define PSK_OP_DIV 0x13
#define PSK_OP_MAX 0x14
#define PSK_OP_MIN 0x15
#define PSK_OP_NEG 0x20
#define PSK_OP_ABS 0x21
#define PSK_OP_EXP 0x22
#define PSK_OP_EXPC 0x23
#define PSK_OP_GELU 0x24
#define PSK_OP_SQRT 0x25
#define PSK_OP_SQRTA 0x26
#define PSK_OP_ERF 0x27
#define PSK_OP_RECIP 0x28
#define PSK_OP_LOG 0x29
#define PSK_OP_TANH 0x2A
#define PSK_OP_SELECT 0x30
#define PSK_MAX_NODES 64
#define PSK_MAX_TOKENS 1024
#define PSK_MAX_INPUTS 16
#define PSK_MAX_IMM 64
#define PSK_MAX_RANK 4

typedef struct {
  const uint32_t* tokens; /* host array of n_tokens tokens */
  int32_t n_tokens;
  const float* imm;       /* host array of n_imm f32 immediates (may be NULL if 0) */
  int32_t n_imm;
} psk_program;

/* An input read through element strides, one per OUTPUT axis (the output's
 * rank): output element (i0, .., i_{r-1}) reads ptr[sum_k i_k * stride[k]].
 * A stride of 0 broadcasts along that axis (a row vector [C] into [R, C] is
 * stride {0, 1}; a column [R, 1] is {1, 0}; a scalar is {0, 0}).  Strides are
 * in elements and must be >= 0. */
typedef struct {
  const void* ptr;
  int32_t dtype;              /* psk_dtype: PSK_F32, PSK_BF16, or PSK_I32 for a SELECT condition */
  int64_t stride[PSK_MAX_RANK];
} psk_input;

/* The root's storage: contiguous row-major, rank 0..4 (rank 0 = one element). */
typedef struct {
  void* ptr;
  int32_t dtype;              /* psk_dtype */
  int32_t rank;
  int64_t shape[PSK_MAX_RANK];
} psk_output;

/* Evaluate the group over every output element, in one launch (several for
 * more than 2^30 vectors of elements) of a kernel generated for this program
 * and compiled at run time on its first use (see psk_group_prepare).  The output may alias an input only
 * if that input has exactly the output's layout (same pointer, dtype and
 * row-major strides): each element is then read before it is written.  Any
 * other overlap is refused with PSK_E_ALIAS when the pointers show it. */
int psk_group_run(const psk_program* prog, const psk_input* inputs, int32_t n_inputs,
                  const psk_output* out, void* stream);

/* Host-only check of a program (no launch, no device needed): returns 0, the
 * number of op nodes and the most values (inputs and node results) one
 * element keeps live at once, or the refusal psk_group_run would give for the
 * program's structure.  Input types (the PSK_I32 rule of SELECT) need the
 * input descriptors and are checked by psk_group_prepare / psk_group_run. */
int psk_group_check(const psk_program* prog, int32_t n_inputs, int32_t* n_nodes, int32_t* n_values);

/* Host-only, synchronous, needs no device: everything psk_group_run does
 * before the launch -- validate the program and the descriptors, and compile
 * (once per process; cached) the kernel specialised for this program, its
 * inputs' storage types and access modes, the vector width and the root's
 * storage type.  Pointers are inspected for alignment and overlap only, never
 * dereferenced.  Lets a caller take the compile (about a second) out of a
 * timed or latency-sensitive region; psk_group_run compiles on first use
 * otherwise.  Returns the refusal psk_group_run would give, or PSK_E_CUDA
 * with the compiler's message. */
int psk_group_prepare(const psk_program* prog, const psk_input* inputs, int32_t n_inputs, const psk_output* out);

/* psk_group_run / psk_group_prepare with a math mode (a psk_exp_mode, below):
 * PSK_EXP_EXACT is psk_group_run itself (every node correctly rounded);
 * PSK_EXP_FAST is a declared fast realization of the EXP, EXPC and ERF
 * nodes: EXP within one f32 ulp, EXPC (the multifunction unit's 2^f after an
 * exact reduction) and ERF within two of the correctly rounded values
 * (measured over their ranges).  GELU, LOG and TANH
 * stay correctly rounded in this mode: gelu's 1 + erf(t) is exact and
 * cancels where erf(t) < -1/2, so any error in erf there is magnified in
 * gelu's result, and only the correctly rounded erf keeps gelu within two
 * ulp.  Not bit-identical to the oracle; on the 64-node workload a few
 * outputs in 10^6 differ, by one bf16
 * ulp.  PSK_E_ARG for another mode; otherwise as psk_group_run. */
int psk_group_run_ex(const psk_program* prog, const psk_input* inputs, int32_t n_inputs,
                     const psk_output* out, int32_t math_mode, void* stream);
int psk_group_prepare_ex(const psk_program* prog, const psk_input* inputs, int32_t n_inputs,
                         const psk_output* out, int32_t math_mode);

/* psk_group_run_ex through one kernel compiled with the library for every
 * program, which walks the program's node list per element (the group as one
 * loop nest whose body is the chain of members, PSK-Realize "What a group
 * is"; each node evaluated as the unfused op would be, presk "Native
 * execution": fusion reassociates nothing).  The same validation, refusals,
 * aliasing rule and result bits as psk_group_run_ex with the same math mode;
 * no run-time compilation, so no first-use compile and no run-time compiler
 * needed; slower than the kernel specialised for the program (the dispatch
 * per node and the values' trips through per-thread local memory), and the
 * baseline that specialisation is measured against.  Asynchronous on the
 * stream; PSK_E_CUDA if the launch fails. */
int psk_group_run_interp(const psk_program* prog, const psk_input* inputs, int32_t n_inputs,
                         const psk_output* out, int32_t math_mode, void* stream);

/* ================================================== psk_softmax_region
 * y[r, :] = softmax(x[r, :]) over rows of `cols` elements: m = max_j x[r,j]
 * (NaN propagates), e_j = exp(x[r,j] - m), s = the sum of e_j in the declared
 * order, y = RN(e_j / s) (IEEE division) rounded to yt.  Orders:
 *   SEQUENTIAL       s = (((e0 + e1) + e2) + ...)
 *   BLOCKED(w)       the same chain (register blocking keeps index order), w >= 1
 *   INTERLEAVED(P)   partial p sums e_j, j = p mod P, in increasing j; the P
 *                    partials are then added left to right; 1 <= P <= 64
 *                    (INTERLEAVED(1) is SEQUENTIAL).
 * exp_mode EXACT uses the correctly rounded exp (bit-identical to a group's EXP
 * node); FAST uses a fast exp (within two f32 ulp of it, the tolerance stated
 * for exp nodes; measured over [-104.5, 0]), a declared realization that owes
 * its measured gap.  x and y are row-major with leading
 * dimensions ldx, ldy >= cols (elements); y must not overlap x unless y == x
 * with the same dtype and leading dimension (in place).  rows or cols == 0 is
 * an empty region (nothing launched, returns 0). */
typedef enum { PSK_ORDER_SEQUENTIAL = 0, PSK_ORDER_BLOCKED = 1, PSK_ORDER_INTERLEAVED = 2 } psk_order_kind;
typedef struct { int32_t kind; int32_t param; } psk_order;
typedef enum { PSK_EXP_EXACT = 0, PSK_EXP_FAST = 1 } psk_exp_mode;

int psk_softmax_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                       int64_t ldx, int64_t ldy, psk_order order, int32_t exp_mode, void* stream);

/* The masked softmax region (presk "Native execution", numerics: a mask is
 * an index buffer of 0 and 1; the masked softmax takes its maximum from the
 * allowed positions and its sum over them, writes 0 where it refuses, and a
 * row it empties gives zeros -- otherwise the bits of the softmax of the
 * scores with -inf at the refused positions).  mask: DEVICE bytes, nonzero
 * allows; ldm = 0 applies one mask row of cols bytes to every row, ldm >= cols
 * gives each row its own.  Other arguments as psk_softmax_region; y must not
 * overlap the mask; cols up to 49152. */
int psk_softmax_masked(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                       int64_t ldx, int64_t ldy, const uint8_t* mask, int64_t ldm, psk_order order,
                       int32_t exp_mode, void* stream);

/* The softmax region's backward (presk "The language", automatic
 * differentiation: softmax's rule is y (ct - sum_axis(ct y))): per row
 * s = sum_j RN(ct_j y_j) in the declared order, dx_j = RN(y_j RN(ct_j - s)),
 * rounded to dxt.  y (the forward's output), ct (the cotangent) and dx are
 * DEVICE rows with leading dimensions ldy, ldc, ldd >= cols; dx may be y or ct
 * in place (same type and leading dimension), no other overlap; cols up to
 * 49152. */
int psk_softmax_backward(const void* y, int32_t yt, const void* ct, int32_t ct_t, void* dx, int32_t dxt,
                         int64_t rows, int64_t cols, int64_t ldy, int64_t ldc, int64_t ldd, psk_order order,
                         void* stream);

/* ==================================================== psk_norm_region
 * The normalization regions over rows of `cols` elements, each a last-axis
 * reduction and its pointwise epilogue in one launch (poot "Fusion and
 * Planning", Reduction-rooted regions: RMSNorm is sum-of-squares -> sqrt ->
 * div; presk PSK-Realize, "What it removes": the layer normalization chain
 * (x - mu)^2 -> mean -> +eps -> sqrt -> divide).  In f32, one rounding per
 * operation, n = cols, eps rounded once to f32, every sum in the declared
 * order (as psk_softmax_region's):
 *   RMSNorm   ss = sum RN(x_j^2); d = sqrt(RN(RN(ss / n) + eps));
 *             y_j = RN(x_j / d) [then RN(. * gamma_j)]
 *   LayerNorm mu = RN(sum x_j / n); c_j = RN(x_j - mu); ss = sum RN(c_j^2);
 *             d = sqrt(RN(RN(ss / n) + eps));
 *             y_j = RN(c_j / d) [then RN(. * gamma_j)] [then RN(. + beta_j)]
 * Divisions and sqrt are IEEE.  gamma and beta are DEVICE vectors of cols
 * elements of param_dtype (f32 or bf16, widened exactly), or NULL for none;
 * RMSNorm takes no beta.  x, y, ldx, ldy, rows, cols and in-place use as in
 * psk_softmax_region; y must not overlap gamma or beta.  cols up to 49152;
 * eps must be finite. */
typedef enum { PSK_NORM_RMS = 0, PSK_NORM_LAYER = 1 } psk_norm_kind;

int psk_norm_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                    int64_t ldx, int64_t ldy, int32_t kind, double eps, const void* gamma, const void* beta,
                    int32_t param_dtype, psk_order order, void* stream);

/* ====================================================== psk_adamw_tree
 * One AdamW step over every leaf, in place, one launch for the whole tree
 * (trees of more than PSK_ADAMW_MAX_LEAVES leaves take one launch per that
 * many leaves).  Per parameter, in f32, one rounding per operation:
 *   m' = (b1 m) + ((1-b1) g);  v' = (b2 v) + ((1-b2) (g g))
 *   m^ = m' / (1-b1^t);  v^ = v' / (1-b2^t)
 *   theta' = theta - lr ((m^ / (sqrt(v^) + eps)) + wd theta)
 * The scalars b1, b2, 1-b1, 1-b2, 1-b1^t, 1-b2^t, lr, eps, wd are computed
 * from the binary64 hyperparameters on the host and rounded once to f32
 * (psk_adamw_scalars returns them).  theta, m, v are f32, or bf16 per leaf
 * (param_dtype); grad is f32 or bf16 (widened exactly).  t >= 1;
 * 0 < beta < 1; leaves must not overlap. */
#define PSK_ADAMW_MAX_LEAVES 512
typedef struct {
  void* theta;          /* param_dtype */
  void* m;              /* param_dtype */
  void* v;              /* param_dtype */
  const void* grad;
  int32_t grad_dtype;   /* psk_dtype */
  int32_t param_dtype;  /* psk_dtype of theta, m and v: PSK_F32 (0, the default) or PSK_BF16, a leaf stored in
                           bf16 at rest (presk "Native execution", params): widened exactly, stepped in f32,
                           each of theta', m', v' rounded once to bf16 */
  int64_t numel;        /* >= 0; 0 skips the leaf */
} psk_leaf;
typedef struct { double lr, beta1, beta2, eps, weight_decay; int64_t t; } psk_adamw_hparams;

int psk_adamw_tree(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp, void* stream);

/* Host-only: the nine f32 scalars the step reads, in the order
 * b1, b2, 1-b1, 1-b2, 1-b1^t, 1-b2^t, lr, eps, wd (constant schedule). */
int psk_adamw_scalars(const psk_adamw_hparams* hp, float out[9]);

/* ---------------------------------------------- schedules and clipping
 * presk "The language", The optimizer: with grad_clip = c the gradient is
 * first scaled by min(1, c / (||g||_2 + 1e-6)), the global norm over the tree;
 * schedules constant(), linear(warmup = w) -- lr t/w for t <= w, then
 * lr (total - t)/(total - w) -- and cosine(warmup = w) -- lr t/w, then
 * lr 1/2 (1 + cos(pi (t - w)/(total - w))) -- both 0 from t = total on.
 * The scheduled lr is computed exactly from the binary64 arguments and
 * rounded once to f32 (psk_adamw_lr returns it).  Clipping (grad_clip > 0):
 *   ||g||^2 = f32 sum of RN(g^2) over a declared tree -- blocks of 1024
 *   consecutive elements of a leaf (in order), groups of 64 blocks (in
 *   order), a leaf's groups (in order), the leaves (in order; empty leaves
 *   skipped);
 *   q = RN(c / RN(sqrt(||g||^2) + RN(1e-6))), scale = q < 1 ? q : 1;
 *   every gradient enters the step as RN(g * scale).
 * warmup 0 has no warmup piece; linear and cosine need
 * 0 <= warmup < total < 2^52; grad_clip must be finite, 0 = no clipping. */
typedef enum { PSK_LR_CONSTANT = 0, PSK_LR_LINEAR = 1, PSK_LR_COSINE = 2 } psk_lr_kind;
typedef struct {
  int32_t kind;         /* psk_lr_kind */
  int64_t warmup, total;
  double grad_clip;     /* c; 0 = none */
} psk_adamw_schedule;

/* Host-only: the scheduled f32 lr of step hp->t. */
int psk_adamw_lr(const psk_adamw_hparams* hp, const psk_adamw_schedule* sched, float* lr);

/* Host-only: the DEVICE workspace bytes psk_adamw_tree_ex needs for these
 * leaves and this schedule (0 without clipping: about 4 bytes per 1024
 * parameters with it). */
int psk_adamw_workspace(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_schedule* sched,
                        uint64_t* bytes);

/* psk_adamw_tree with a schedule (NULL: constant, no clipping) and, when
 * clipping, a caller-owned 16-byte aligned DEVICE workspace of at least
 * psk_adamw_workspace bytes (its contents need no initialisation and are
 * scratch: concurrent calls must not share one).  Clipping adds three short
 * launches (the squared-norm tree and the scale) before the update. */
int psk_adamw_tree_ex(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                      const psk_adamw_schedule* sched, void* workspace, uint64_t workspace_bytes, void* stream);

/* psk_adamw_tree_ex without a caller workspace: when clipping, its scratch
 * is a fixed buffer of PSK_ADAMW_STATIC_WORKSPACE bytes inside the library's
 * device module (one per device, reserved when the module loads), so the call
 * allocates nothing: no device memory (no cudaMalloc, no caller workspace)
 * and no host heap (its kernel-parameter staging is per host thread, reused
 * from call to call).  The pages have no counterpart: it exists for callers
 * that cannot hand the library device memory -- code whose device memory
 * belongs to another allocator (a framework's pool that holds it all), or
 * that must not fail for lack of memory in the middle of a training step.
 * The buffer's device
 * address is looked up on the first call per device and CUDA context (the
 * set-up runs with that device current; make the first call before any stream
 * capture).  Limits: trees whose clipping scratch exceeds the buffer (about
 * 2 * 10^9 parameters) are refused with PSK_E_ARG; calls that overlap in time
 * on one device (other streams, other threads) share the buffer and race, so
 * they must be serialised (one stream, or events).  Without clipping it is
 * psk_adamw_tree_ex. */
#define PSK_ADAMW_STATIC_WORKSPACE (8u << 20)
int psk_adamw_tree_static(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                          const psk_adamw_schedule* sched, void* stream);

/* ------------------------------------ the clipped step over several ranks
 * presk PSK-Realize, "Memory placement and collectives": a tree split across
 * processes (one per GPU) updates with no exchange, except that clipping
 * needs the global ||g||^2.  Its declared tree (blocks of 1024 elements,
 * groups of 64 blocks, a leaf's groups, the leaves, each in order; see
 * "schedules and clipping") makes the group sums the unit to exchange: a
 * rank whose pieces of leaves start on group boundaries (multiples of 65,536
 * elements of their leaf) computes its pieces' group sums exactly as the
 * one-process step does; gathered in leaf order they give the same ||g||^2,
 * scale and update bits on every rank.  The three calls:
 *
 * psk_adamw_group_sqsums: the group sums of `leaves` (pieces of the tree's
 * leaves, each starting on a group boundary of its leaf), leaf after leaf in
 * order, into group_sums (DEVICE, ceil(ceil(numel / 1024) / 64) floats per
 * non-empty leaf); workspace as for psk_adamw_tree_ex with clipping
 * (psk_adamw_workspace with grad_clip > 0).
 *
 * psk_adamw_clip_scale: from the whole tree's group sums (DEVICE, the
 * gathered lists in leaf order) and the number of groups of each of its
 * n_leaves leaves (HOST array; 0 for an empty leaf; n_leaves <=
 * PSK_ADAMW_MAX_LEAVES), the scale min(1, c / (sqrt(||g||^2) + 1e-6)) into
 * *scale (DEVICE); c = grad_clip > 0, finite.
 *
 * psk_adamw_tree_scaled: psk_adamw_tree_ex on the rank's pieces with every
 * gradient scaled by *scale (DEVICE) as clipping does, the schedule's lr
 * (its grad_clip is not used; NULL: constant lr).
 *
 * Refusals as for psk_adamw_tree_ex (PSK_E_NULL for a NULL scale, group_sums
 * or workspace where one is needed; PSK_E_ARG otherwise).  Asynchronous on
 * the stream; the exchange between the first two calls is the caller's (an
 * all-gather of the group sums). */
int psk_adamw_group_sqsums(const psk_leaf* leaves, int32_t n_leaves, float* group_sums, void* workspace,
                           uint64_t workspace_bytes, void* stream);
int psk_adamw_clip_scale(const float* group_sums, const int64_t* groups_per_leaf, int32_t n_leaves, double grad_clip,
                         float* scale, void* stream);
int psk_adamw_tree_scaled(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                          const psk_adamw_schedule* sched, const float* scale, void* stream);

/* Host-only, synchronous: the device status word of the pipelined kernels of
 * the current device (0 = no bounded wait ever timed out; bit 0 = a wait gave
 * up and the kernel wound down, its output then unspecified).  reset != 0
 * clears the word after reading it.  A timeout is never expected: it would
 * mean a pipeline bug, and this lets a caller detect it without a hang. */
int psk_device_status(uint32_t* status, int32_t reset);

/* Test hook for the bounded waits (no counterpart on the pages): from the
 * next launch on, the pipelined row-region kernels of the current device stop
 * producing at local row `row` of every CTA, as if that row's copy had been
 * lost.  Every wait for it gives up after about two seconds of clock, the
 * kernel sets bit 0 of the status word and winds down (its output then
 * unspecified), and the device stays usable.  row = -1 (the default) turns
 * it off.  Host-only, synchronous; for tests, never for production use.
 * PSK_E_ARG for row < -1. */
int psk_test_drop_row(int64_t row);

/* Test hook for the softmax region's fast realization (presk "Native
 * execution": a realization that approximates owes a measured gap; the exp
 * nodes' tolerance is two f32 ulp): y[i] = the fast exp of x[i], the function
 * the region's fast realization applies to every x - max (x[i] <= 0, NaN or
 * -inf; larger x are outside its domain and give unspecified values), so
 * that tests can measure its bound over whole binades.  x and y: n floats in
 * DEVICE memory (y may be x); asynchronous on the stream.  PSK_E_NULL for a
 * NULL pointer with n > 0, PSK_E_SHAPE for n < 0, PSK_E_CUDA if the launch
 * fails; n = 0 launches nothing.  For tests, never for production use. */
int psk_test_fast_exp(const float* x, float* y, int64_t n, void* stream);

/* Thread-local description of the last refusal of this thread ("" if none). */
const char* psk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PSK_H */
