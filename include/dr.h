/*
 * dr.h — C-ABI of libdr: the generalised gated delta-rule recurrence on one
 * GB300 (sm_103a).
 *
 * The operation (Kalman Delta Networks notes, section 1, unified recurrence and
 * the table under it; Kaczmarz Linear Attention notes, section 1.1 and Eq. (3)):
 *
 *     S~_t = D_t S_{t-1}
 *     e_t  = v_t - S~_t^T k_t
 *     S_t  = S~_t + w_t e_t^T
 *     o_t  = S_t^T q_t                       (read after the write)
 *
 * S_t is a dk x dv fp32 matrix per (batch, head).  D_t = alpha_t I for GDN, KLA
 * and PGDN, diag(alpha_t) (scaling the rows of S) for Diagonal KDN, KDA and
 * PKDA, isotropic KDN, exact Kalman; alpha = exp(log_alpha).  The write vector w_t
 * per variant:
 *
 *   DR_GDN   w = eta k                        (KLA notes section 1.1)
 *   DR_KLA   w = eta k / (||k||^2 + eps)      (KLA notes Eq. (3), Algorithm 1)
 *   DR_PGDN  A_t = alphaP A_{t-1} + betaP (k*k);  r = ln max(A_t, log_floor) - mu;
 *            B = exp(-ln(x) r / (1 + |r|));  w = eta (B * k)
 *                                             (Preconditioned DeltaNet notes Eq. (9))
 *   DR_KDN   p^ = alpha^2 p_{t-1} + omega;  kappa = p^ k / (r + sum p^ k^2);  w = kappa;
 *            p_t = p^ / (1 + (info_scale / r) k*k p^)
 *                                             (KDN notes Eqs. (23)-(30), (60)-(65))
 *   DR_KDA   w = eta k with per-channel decay (KDN notes section 1, table)
 *   DR_PKDA  the DR_PGDN write key with per-channel decay
 *                                             (Preconditioned DeltaNet notes section 2.5)
 *   DR_IKDN  isotropic KDN, one variance b per head, per-channel decay:
 *            a = mean_i alpha_i^2;  b^ = a b_{t-1} + omega;  w = b^ k / (r + b^ ||k||^2);
 *            b_t = b^ / (1 + info_scale ||k||^2 b^ / (dk r))
 *                                             (KDN notes section 7, Eq. (40))
 *   DR_EKDN  exact Kalman memory, dense key covariance P (dk x dk), per-channel decay:
 *            P^ = D P D^T + diag(omega);  w = P^ k / (r + k^T P^ k);  P_t = (I - w k^T) P^
 *                                             (KDN notes section 2.2, Eqs. (12)-(17));
 *            token by token (no chunked form; `chunk` is checked but unused); P_0
 *            must be symmetric (a covariance), which every update preserves
 *
 * q and k are L2-normalised first when the corresponding flag is set
 * (q / max(||q||, 1e-30)); KLA reads out with the normalised query (KLA notes
 * Eq. (3)).  "k" above is then the normalised key everywhere.
 *
 * Layouts (row-major, innermost index last):
 *   q, k     [B, T, H, dk]      v, out [B, T, H, dv]     (decode: T absent)
 *   log_alpha [B, T, H]  (KDN, KDA, PKDA, IKDN, EKDN: [B, T, H, dk])
 *   eta, alphaP, betaP, r [B, T, H];  omega [B, T, H, dk] (IKDN [B, T, H]);  mu [H]
 *   state    [B, H, dk, dv] fp32;  aux (PGDN / PKDA A, KDN p) [B, H, dk] fp32,
 *            (IKDN b) [B, H] fp32, (EKDN P) [B, H, dk, dk] fp32
 * q/k/v/out are fp32 (DR_FP32) or bf16 (DR_BF16); every gate and state is fp32.
 *
 * Ownership: the caller owns every buffer; all pointers are device pointers
 * unless stated otherwise.  The library allocates no device memory and never
 * synchronises except in dr_get_device_status().  Calls are asynchronous on
 * `stream` and may be captured in a CUDA graph.
 *
 * Errors: argument problems return a negative dr_status before anything is
 * launched.  A launch failure returns DR_ERR_CUDA.  Problems found on the
 * device (non-finite values when check_finite is set, a bounded wait that ran
 * out) set a sticky device status word that dr_get_device_status() returns.
 * Nothing traps.
 */
#ifndef DR_H
#define DR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dr_stream_t;

typedef enum {
  DR_GDN = 0, DR_KLA = 1, DR_PGDN = 2, DR_KDN = 3, DR_KDA = 4, DR_PKDA = 5, DR_IKDN = 6,
  DR_EKDN = 7
} dr_variant;

typedef enum { DR_FP32 = 0, DR_BF16 = 1 } dr_dtype;

typedef enum {
  DR_OK = 0,
  DR_ERR_NULL = -1,        /* a required pointer is NULL                         */
  DR_ERR_SHAPE = -2,       /* unsupported size (see each call)                   */
  DR_ERR_DTYPE = -3,       /* dtype not DR_FP32 / DR_BF16                        */
  DR_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned                   */
  DR_ERR_WORKSPACE = -5,   /* workspace missing or too small                     */
  DR_ERR_CUDA = -6,        /* a CUDA call or launch failed                       */
  DR_ERR_TIMEOUT = -7,     /* a bounded device-side wait gave up                 */
  DR_ERR_NONFINITE = -8,   /* check_finite found NaN/Inf in an output            */
  DR_ERR_UNSUPPORTED = -9, /* variant / option combination not implemented       */
  DR_ERR_ARG = -10         /* a scalar argument is out of range                  */
} dr_status;

/* Gate parameters shared by both calls.  Unused fields may be NULL / ignored.
 * Initialise with dr_params_init() and set what the variant needs. */
typedef struct dr_params {
  int dtype;               /* dr_dtype of q, k, v and out                             */
  int q_l2norm;            /* 1: normalise q before reading out                       */
  int k_l2norm;            /* 1: normalise k before the residual and the write        */
  const float *eta;        /* GDN/KLA/KDA eta, PGDN/PKDA beta: [B,T,H] (decode [B,H]) */
  const float *alphaP;     /* PGDN/PKDA statistic decay [B,T,H] (decode [B,H])        */
  const float *betaP;      /* PGDN/PKDA statistic gain  [B,T,H] (decode [B,H])        */
  const float *mu;         /* PGDN/PKDA per-head centre [H]                           */
  float x;                 /* PGDN bound, B in [1/x, x]; default 1.5                  */
  float log_floor;         /* PGDN guard: ln max(A, log_floor); default 1e-12         */
  const float *omega;      /* KDN/EKDN process noise [B,T,H,dk] (decode [B,H,dk]); IKDN [B,T,H] */
  const float *r;          /* KDN/IKDN observation noise [B,T,H] (decode [B,H]), > 0  */
  float info_scale;        /* KDN/IKDN information scaling mu; default 1 (strict)     */
  const float *aux_init;   /* dr_chunk_fwd: PGDN/PKDA A_0, KDN p_0 [B,H,dk], IKDN b_0
                              [B,H], EKDN P_0 [B,H,dk,dk]; NULL => 0, 1, 1, I          */
  float *aux_final;        /* dr_chunk_fwd: final A / p [B,H,dk]; NULL => not written */
  void *workspace;         /* dr_chunk_fwd: caller-owned device scratch, 256-byte     */
  size_t workspace_bytes;  /* aligned, or NULL (see dr_chunk_fwd_workspace_bytes)     */
  int check_finite;        /* 1: scan outputs/states for NaN/Inf -> DR_ERR_NONFINITE  */
} dr_params;

/* Fill *p with the defaults above (dtype DR_BF16, x 1.5, log_floor 1e-12,
 * info_scale 1, everything else 0/NULL). */
void dr_params_init(dr_params *p);

/*
 * Chunkwise-parallel forward over a whole sequence (prefill / training forward).
 *
 * Computes exactly the recurrence above for t = 1..T from init_state, chunk by
 * chunk: within a chunk the tokens' mutual dependence is the unit
 * lower-triangular system [I + L] E = V - (Gamma.K) S_0 with
 * L_ij = sum_c k_ic w_jc exp(g_ic - g_jc) (j < i), solved on chip, then
 * O = (Gamma.Q) S_0 + P E and S_out = diag(gamma_C) S_0 + (exp(g_C - g_j).W)^T E
 * (KLA notes section 2.5, Eqs. (7)-(9), generalised to a write matrix W as in
 * the Preconditioned DeltaNet notes, section 2.6).  The result is the same as
 * the tokenwise recurrence up to rounding for any chunk size.
 *
 * q, k, v, out     device, dtype gp->dtype, layouts above, 16-byte aligned.
 * log_alpha        device fp32 [B,T,H] (KDN: [B,T,H,dk]).
 * gp               host pointer; its device pointers must match the variant.
 * variant          dr_variant.  eps: KLA stabiliser (>= 0).
 * init_state       device fp32 [B,H,dk,dv] or NULL (zero state).
 * final_state      device fp32 [B,H,dk,dv] or NULL (not written).
 * Sizes: B, H, T >= 1; dk, dv in {64, 128}; chunk in {16, 32, 64, 128}.  T need
 * not be a multiple of chunk.
 * gp->workspace    optional.  Where dr_chunk_fwd_workspace_bytes() is non-zero
 *                  and a workspace of at least that size is given, the
 *                  chunk-local work (Grams, gates, triangular inverse, W') of
 *                  all chunks runs first, in parallel, and leaves one record per
 *                  chunk there; the carry over chunks then reads them.  Its
 *                  contents are undefined afterwards.  NULL: the single-kernel
 *                  path runs (same results up to rounding order).  A workspace
 *                  that is too small returns DR_ERR_WORKSPACE, a misaligned one
 *                  DR_ERR_ALIGN.  Two calls in flight must not share one.
 * Returns DR_OK or a negative dr_status.
 */
int dr_chunk_fwd(const void *q, const void *k, const void *v, const float *log_alpha,
                 const dr_params *gp, int variant, float eps,
                 const float *init_state, void *out, float *final_state,
                 int B, int T, int H, int dk, int dv, int chunk, dr_stream_t stream);

/*
 * One tokenwise step for every (batch, head) (decode).  Reads the state once
 * and writes it once, in place; o = S_t^T q = alpha S^T q + (w^T q) e is formed
 * from the same read (KLA notes Algorithm 1; PDN notes section 2.5; KDN notes
 * section 2.2, predict -> gain -> update -> read).
 *
 * q, k [B,H,dk]; v, out [B,H,dv] (dtype gp->dtype); log_alpha [B,H] (KDN,
 * KDA, PKDA, IKDN, EKDN [B,H,dk]); gate arrays without the T axis.  state
 * [B,H,dk,dv] fp32 in/out.  aux_state fp32 in/out, required for the variants
 * that carry one, ignored otherwise: PGDN / PKDA A or KDN p [B,H,dk], IKDN b
 * [B,H], EKDN P [B,H,dk,dk] (the exact Kalman step runs one CTA per head and
 * updates state and P in place).  gp->aux_init/aux_final are ignored.
 * Sizes: B, H >= 1; dk, dv in {64, 128}.
 */
int dr_decode_step(const void *q, const void *k, const void *v, const float *log_alpha,
                   const dr_params *gp, int variant, float eps,
                   float *state, float *aux_state, void *out,
                   int B, int H, int dk, int dv, dr_stream_t stream);

/* Bytes of the optional dr_chunk_fwd workspace for these sizes: B H ceil(T/64)
 * records on the two-phase paths (dk = dv = 128, chunk 64) of 66560 bytes (GDN,
 * KLA; bf16), 101376 bytes (PGDN, bf16: also the write keys and the key
 * statistic's chunk map and chunk-start value) or 135168 bytes (Diagonal KDN,
 * KDA and PKDA, bf16 or fp32: the carry's operands -- bf16 hi/lo tile images
 * for bf16 inputs, fp32 for fp32 -- and the variance / statistic chunk map and
 * chunk-start value), plus for those three 4 (n + 2) bytes rounded up to 256
 * (n = B H ceil(T/64) records): the flags of the chain between chunks, which
 * the call clears itself; 0 where no path uses one.  On the GDN / KLA / PGDN
 * path, when the rows are few against the current device's SM count (6 B H <=
 * SMs) and the rows long, the carry is cut into G segments run in parallel and
 * the workspace adds 3 B H G x 64 KB for the segments' end states, transition
 * maps and start states (G depends on the SM count: query on the device that
 * runs the call). */
size_t dr_chunk_fwd_workspace_bytes(int variant, int dtype, int B, int T, int H, int dk, int dv,
                                    int chunk);

/*
 * Same forward as dr_chunk_fwd on its two-phase paths (GDN, KLA, PGDN in bf16
 * and Diagonal KDN, KDA, PKDA, isotropic KDN in bf16 or fp32; dk = dv = 128, chunk 64), for callers that
 * cannot allocate device
 * memory: code that runs where cudaMalloc is off limits (a host framework that
 * owns every byte of device memory through its own allocator, a real-time loop
 * that must not take cudaMalloc's implicit device synchronisation, a plug-in
 * handed only its input and output buffers).  The paper has no counterpart:
 * this is an interface convenience, not part of the method.
 *
 * The per-chunk records live in one library-owned device array of
 * DR_NOALLOC_SCRATCH_BYTES, created with the library's CUDA module on every
 * device that loads it and held until the process exits.  The caller still
 * passes every input and output; gp->workspace is ignored.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it with the
 *     current context; make that first call before any stream capture.  A new
 *     context on the device (after cudaDeviceReset) gets a new array, whose
 *     address the next call looks up again (again outside any capture).
 *   - Argument checks come first, in dr_chunk_fwd's order (DR_ERR_NULL,
 *     DR_ERR_DTYPE, DR_ERR_SHAPE), then the path and size checks below.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind (nothing in it has to start at zero).  Calls that overlap on the
 *     GPU -- two streams, or two host threads -- race on it: serialise them.
 * Returns DR_ERR_UNSUPPORTED for other variants, dtypes or shapes (dr_chunk_fwd
 * needs no workspace for those), DR_ERR_WORKSPACE when the workspace
 * (dr_chunk_fwd_workspace_bytes) would exceed DR_NOALLOC_SCRATCH_BYTES: about
 * B H ceil(T/64) > 1008 records (GDN, KLA), > 661 (PGDN) or > 496 (KDN, KDA,
 * PKDA, IKDN), fewer when the segment area of a few-row call is added;
 * otherwise whatever dr_chunk_fwd returns.
 */
#define DR_NOALLOC_SCRATCH_BYTES (64u << 20)
int dr_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                         const dr_params *gp, int variant, float eps,
                         const float *init_state, void *out, float *final_state,
                         int B, int T, int H, int dk, int dv, int chunk, dr_stream_t stream);

/* Synchronises `stream`, returns and clears the sticky device status
 * (DR_OK, DR_ERR_NONFINITE or DR_ERR_TIMEOUT), or DR_ERR_CUDA. */
int dr_get_device_status(dr_stream_t stream);

/* Gradient buffers of dr_chunk_bwd (device fp32, overwritten; NULL where a
 * field says so).  Layouts as the forward's inputs. */
typedef struct dr_grads {
  float *dq;               /* [B,T,H,dk]                                              */
  float *dk;               /* [B,T,H,dk]                                              */
  float *dv;               /* [B,T,H,dv]                                              */
  float *d_log_alpha;      /* [B,T,H]; per-channel decay (KDA, KDN): [B,T,H,dk]      */
  float *d_eta;            /* [B,T,H] (GDN / KLA eta, PGDN beta, KDA eta); KDN: NULL  */
  float *d_init_state;     /* [B,H,dk,dv] or NULL (not written)                       */
  float *d_alphaP;         /* PGDN: [B,T,H]                                           */
  float *d_betaP;          /* PGDN: [B,T,H]                                           */
  float *d_mu;             /* PGDN: [H]                                               */
  float *d_aux_init;       /* PGDN: dL/dA_0, Diagonal KDN: dL/dp_0 [B,H,dk] or NULL   */
  const float *d_aux_final;/* PGDN: input dL/dA_T, KDN dL/dp_T [B,H,dk] or NULL (zero) */
  float *d_omega;          /* Diagonal KDN: [B,T,H,dk]                                */
  float *d_r;              /* Diagonal KDN: [B,T,H]                                   */
} dr_grads;

/*
 * Backward of dr_chunk_fwd (training): given dL/d out, dL/d final_state (and for
 * PGDN dL/d A_T), the gradients of L with respect to q, k, v, log_alpha, the
 * write gates and init_state (PGDN also alphaP, betaP, mu and A_0), for the
 * scalar-decay write rules GDN, KLA and PGDN (KLA notes section 2.5, Eqs.
 * (7)-(9) differentiated chunk by chunk in reverse; then the write gain: GDN /
 * KLA section 1.1 / Eq. (3); PGDN the bounded map of the key statistic, PDN
 * notes Eq. (9), whose adjoint is carried backwards through the statistic's
 * recursion; then the optional L2 norms).  The forward is run again inside the
 * call (its chunk records, the state at every chunk start and the chunk
 * residuals E go to the workspace); a reverse carry over chunks passes dL/dS
 * from chunk to chunk, and every chunk's local gradients follow in parallel.
 *
 * Inputs as dr_chunk_fwd (same q, k, v, log_alpha, gp gates and flags --
 * gp->aux_init is PGDN's A_0 --, eps, init_state or NULL).  d_out [B,T,H,dv] in
 * gp->dtype; d_final_state fp32 [B,H,dk,dv] or NULL (zero).  g: host pointer to
 * the gradient buffers (the PGDN fields are ignored for GDN / KLA).
 * gp->workspace must hold at least dr_chunk_bwd_workspace_bytes() (256-byte
 * aligned); its contents are undefined afterwards.  Supported: DR_GDN, DR_KLA,
 * DR_PGDN with bf16 q/k/v, dk = dv = 128, chunk 64 (DR_ERR_UNSUPPORTED
 * otherwise).  Returns DR_OK or a negative dr_status (DR_ERR_WORKSPACE when the
 * workspace is missing or small).
 */
int dr_chunk_bwd(const void *q, const void *k, const void *v, const float *log_alpha,
                 const dr_params *gp, int variant, float eps, const float *init_state,
                 const void *d_out, const float *d_final_state, const dr_grads *g,
                 int B, int T, int H, int dk, int dv, int chunk, dr_stream_t stream);

/* Workspace bytes dr_chunk_bwd needs, each array on a 256-byte boundary: per
 * chunk record (n = B H ceil(T/64)) the forward's record (66,560 bytes; PGDN
 * 101,376), the chunk-start state (65,536), E (32,768), dL/dS at the chunk end
 * (65,536) and three per-chunk products (32,768 + 2 x 16,384), 4 bytes of
 * gamma <dS, S_c>; PGDN also dL/dw (32,768) and the key-norm factors (256) per
 * record and 4 B H bytes; 0 where the backward is not supported. */
size_t dr_chunk_bwd_workspace_bytes(int variant, int dtype, int B, int T, int H, int dk, int dv,
                                    int chunk);

/*
 * TEST ONLY -- failure injection on the host side of a device wait.  The
 * chained prep of the per-channel-decay two-phase path (Diagonal KDN, PKDA,
 * isotropic KDN with 3 B H >= SM count) hands each row's gain state from a
 * chunk's task to the next one through a flag per record (record index
 * b H ceil(T/64) + h ceil(T/64) + chunk), and a task waits for its flag at most
 * a bounded time.  This call makes the task that would raise flag
 * `withhold_flag` skip it (-1: none; chunk 0 of a row has no flag) and sets the
 * wait's limit to `wait_ns` (> 0; the default is 2e9).  The waiting task then
 * gives up: dr_get_device_status() returns DR_ERR_TIMEOUT, every other waiter
 * is released, the kernels run to their ends (the affected outputs are
 * garbage) and the context stays usable.  Restore with (-1, 2000000000).
 * Synchronous with respect to the host; it affects every later launch on the
 * current device.  The pages have no counterpart: this exists only to test the
 * give-up path.  Returns DR_OK, DR_ERR_ARG or DR_ERR_CUDA.
 */
int dr_set_chain_fault_for_testing(long long withhold_flag, unsigned long long wait_ns);

/* Static, NUL-terminated description of a dr_status value. */
const char *dr_status_string(int status);

/* Name of the kernel path dr_chunk_fwd takes for these arguments; static string.
 * "tc_split" two-phase tcgen05 path (GDN, KLA, PGDN; bf16, dk = dv = 128, chunk 64)
 *          when the workspace of dr_chunk_fwd_workspace_bytes() is supplied;
 *          without a workspace the same shapes take
 * "tc_ws"  the warp-specialised single-kernel tcgen05 path (GDN, KLA), or
 * "tc"     the phase-sequential tcgen05 kernel (PGDN)
 * "tc_pc_split" two-phase per-channel-decay path (Diagonal KDN, KDA, PKDA,
 *          isotropic KDN; bf16, dk = dv = 128, chunk 64) when the workspace is
 *          supplied: every chunk's local work in a tcgen05 prep (the KDN
 *          variance, PKDA key statistic or isotropic variance at each chunk
 *          start handed over between chunks; with few rows, 3 B H < SM count,
 *          Diagonal KDN takes chunk maps and a scan instead and PKDA / isotropic
 *          KDN the fused kernel), then the tcgen05 state carry
 * "simt_split" the same two phases for fp32 inputs on fp32 CUDA cores
 * "simt"   fp32 CUDA-core kernel (everything else: fp32 mode, KDN / KDA / PKDA
 *          without a workspace, dk or dv 64, other chunk sizes)
 * "kalman" the exact Kalman memory, token by token (DR_EKDN, any shape). */
const char *dr_chunk_fwd_path(int variant, int dtype, int dk, int dv, int chunk);

#ifdef __cplusplus
}
#endif

#endif /* DR_H */
