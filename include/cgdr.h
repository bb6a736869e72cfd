/*
 * cgdr.h -- C ABI of libcgdr, the channelwise gated delta rule for GB300 (sm_103a).
 *
 * The operation (per batch b and v-head h, an fp32 state S of shape dk x dv):
 * for each token t,
 *     qn = q_t / sqrt(|q_t|^2 + eps) * q_scale        kn = k_t / sqrt(|k_t|^2 + eps)
 *     S  <- Diag(exp(g_t)) S                           (per key-channel decay)
 *     S  <- S + beta_t kn (v_t - S^T kn)^T             (rank-one delta-rule write)
 *     o_t = S^T qn                                     (read after the write)
 * Sources: the two-traversal token recurrence of "Two-pass optimization for
 * channelwise gated delta rule kernel" (executorch PR #21020, Summary); the
 * fused decode of "Add fused GatedDeltaNet decode Triton kernel" (executorch
 * PR #18865, description: Q/K/V split, L2 norm, head repeat, gating and state
 * update in one kernel); and the routing and chunked form of "Add parallel
 * chunked prefill for channelwise gated delta rule" (executorch PR #21061,
 * Summary: T == 1 uses the token recurrence, T != 1 a chunkwise WY/UT form).
 *
 * Conventions shared by both calls
 *  - All tensor pointers are DEVICE pointers.  Strides are in ELEMENTS; the
 *    innermost dimension (dk or dv) must be contiguous.
 *  - Head repeat: v-head h reads q/k head h / (Hv/Hk) (repeat-interleave;
 *    the pages say only "head repeat").  Hv must be a multiple of Hk.
 *  - Gate, CGDR_GATE_CHANNEL: g [B,T,Hv,dk] fp32 per-channel log-decay and
 *    beta [B,T,Hv] fp32.  CGDR_GATE_GDN (scalar GatedDeltaNet gate):
 *    a, b [B,T,Hv] in `dtype`, A_log and dt_bias [Hv] fp32;
 *    g = -exp(A_log[h]) * softplus(a + dt_bias[h]) for every channel,
 *    beta = sigmoid(b); softplus(x) = x for x > 20.
 *  - state: fp32 [B,Hv,dk,dv], dense (dv fastest), updated in place.
 *    A zero-filled state is the zero initial state.
 *  - o: [B,T,Hv,dv] in `o_dtype` (fp32 or bf16, independent of the input
 *    dtype), accumulated in fp32.  The pages do not fix the output type; a
 *    bf16 o carries up to half a bf16 ulp of rounding on top of the
 *    computation.
 *  - q, k, v, o: 16-byte aligned base pointers; batch/token/head strides
 *    multiples of 8 elements (bf16) or 4 elements (fp32), by each tensor's
 *    own dtype.  g: 16-byte
 *    aligned, strides multiples of 4.  state: 16-byte aligned.
 *  - No input may alias `state` or `o`.
 *
 * Ownership and threading: the caller owns every buffer and the stream.
 * The library allocates no device memory and keeps no mutable global state
 * that changes results: the kernel choice travels in each call's argument
 * block, and the only library-wide data are per-device caches of launch
 * attributes and, for cgdr_prefill_noalloc, its static scratch area (calls of
 * that entry point whose kernels overlap on the GPU race on it).  Calls are
 * safe from several host threads, are asynchronous on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and launch on the calling
 * thread's current device.
 *
 * Errors: arguments are checked on the host before any launch; a failing
 * check returns its code and launches nothing.  CGDR_ERR_CUDA reports a
 * launch error (cudaGetLastError after the launch).  Device faults surface
 * asynchronously, as with any CUDA kernel.  No C++ exception crosses this ABI.
 */
#ifndef CGDR_H_
#define CGDR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CGDR_ABI_VERSION 2

typedef enum cgdr_status {
    CGDR_OK = 0,
    CGDR_ERR_INVALID_ARG = 1,   /* null pointer, negative size, Hv % Hk != 0, T != 1 for decode */
    CGDR_ERR_UNSUPPORTED = 2,   /* dk, dv or chunk outside the supported set, unknown dtype/gate */
    CGDR_ERR_ALIGNMENT = 3,     /* misaligned pointer, stride or non-unit inner stride */
    CGDR_ERR_WORKSPACE = 4,     /* workspace smaller than cgdr_prefill_workspace_size() */
    CGDR_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    CGDR_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (reported through a status word) */
    CGDR_ERR_BOUNDS = 7,        /* debug build only: a device-side index check failed (through a status
                                   word); the access was skipped */
    CGDR_ERR_RANGE = 8          /* a tensor-core prefill met a value of magnitude above 65504 in one of
                                   its fp16 operands (v, the triangular transform, U, or a
                                   decay-scaled key or query when g > 0 grows them); reported through
                                   the status words, the outputs are then invalid: run that call with
                                   CGDR_PREFILL_SIMT */
} cgdr_status;

typedef enum cgdr_dtype { CGDR_F32 = 0, CGDR_BF16 = 1 } cgdr_dtype;
typedef enum cgdr_gate { CGDR_GATE_CHANNEL = 0, CGDR_GATE_GDN = 1 } cgdr_gate;

/* One argument block for both calls.  Zero-initialise it, then fill in. */
typedef struct cgdr_args {
    int32_t B, T, Hk, Hv, dk, dv;   /* dk, dv in {32, 64, 128}; T == 1 for decode */
    int32_t dtype;                  /* cgdr_dtype of q, k, v (and a, b) */
    int32_t gate;                   /* cgdr_gate */
    int32_t l2norm_qk;              /* nonzero: L2-normalise q and k (the usual setting) */
    int32_t chunk;                  /* prefill chunk length 16, 32 or 64; 0 selects 64 */
    int32_t o_dtype;                /* cgdr_dtype of o; zero-initialised = CGDR_F32 */
    int32_t prefill_path;           /* cgdr_prefill_path of this call; zero-initialised = automatic */
    int32_t wait_polls;             /* polls before a bounded device wait on the kernel's own data
                                       gives up; 0 selects 2^20.  A negative value is a test hook for
                                       the failure path: the first such wait of every block is made
                                       on a barrier that nothing completes and gives up after
                                       -wait_polls polls.  After a wait gives up, copies still in
                                       flight are waited for with the default limit before the
                                       kernel exits */
    float q_scale;                  /* applied to q after the norm; <= 0 selects 1/sqrt(dk) */
    float eps;                      /* added to |x|^2 in the L2 norm; < 0 selects 1e-6 */
    const void *q;     int64_t q_sb, q_st, q_sh;        /* [B,T,Hk,dk] */
    const void *k;     int64_t k_sb, k_st, k_sh;        /* [B,T,Hk,dk] */
    const void *v;     int64_t v_sb, v_st, v_sh;        /* [B,T,Hv,dv] */
    const float *g;    int64_t g_sb, g_st, g_sh;        /* [B,T,Hv,dk] (CHANNEL) */
    const float *beta; int64_t beta_sb, beta_st, beta_sh; /* [B,T,Hv]   (CHANNEL) */
    const void *a;     int64_t a_sb, a_st, a_sh;        /* [B,T,Hv]    (GDN) */
    const void *b;     int64_t b_sb, b_st, b_sh;        /* [B,T,Hv]    (GDN) */
    const float *A_log;                                 /* [Hv]        (GDN) */
    const float *dt_bias;                               /* [Hv]        (GDN) */
    float *state;                                       /* [B,Hv,dk,dv] in/out */
    void *o;           int64_t o_sb, o_st, o_sh;        /* [B,T,Hv,dv] out, o_dtype */
    int32_t *status;   /* optional DEVICE int32: a kernel whose bounded wait gave up stores
                          CGDR_ERR_TIMEOUT here, a tensor-core prefill whose fp16 operand left
                          the fp16 range CGDR_ERR_RANGE (its outputs are then invalid).  The library never
                          clears it: zero it before the calls it should cover.  NULL: not reported
                          (the prefill workspace keeps its own status word either way) */
} cgdr_args;

/* ABI version of the loaded library (CGDR_ABI_VERSION it was built with). */
int cgdr_abi_version(void);

/* Static, human-readable name of a status code; never NULL. */
const char *cgdr_status_string(int status);

/*
 * Host-only check of `args` for cgdr_decode (for_prefill == 0) or
 * cgdr_prefill (for_prefill != 0), without touching the GPU.  Returns the
 * status the call itself would return before launching.
 */
cgdr_status cgdr_validate(const cgdr_args *args, int for_prefill);

/*
 * One decode step (T == 1) for every (b, h): the fused path of "Add fused
 * GatedDeltaNet decode Triton kernel" (Q/K/V split by strides into one packed
 * projection row, L2 norm, head repeat, gate, state update, all in one
 * kernel) with the two-traversal update of "Two-pass optimization for
 * channelwise gated delta rule kernel": one pass forms S^T(exp(g) * kn) from
 * the state as read, the other decays, writes and accumulates o.  Each
 * state element is read once from and written once to HBM.
 * The token-stride fields (q_st, ...), chunk and prefill_path are ignored.
 * A state tile whose copy into shared memory never completes (a bounded wait
 * gives up) leaves that tile's state untouched, sets o of every (b, h) the
 * affected block had not finished to NaN and stores CGDR_ERR_TIMEOUT in
 * `status` when that is given.
 */
cgdr_status cgdr_decode(const cgdr_args *args, void *stream);

/*
 * Bytes of device workspace cgdr_prefill needs for `args` (may be 0): 0 for
 * the CUDA-core kernel, 256 for the per-head tensor-core kernel (a status
 * word), 256 + B * Hv * 741888 for the cluster kernel (the status word,
 * then nine 82432-byte hand-off slots per (batch, v-head)), and
 * 256 + ceil256(64 * B * Hv) + B * Hv * 659456 for the cooperative kernel (the
 * status word, 16 sequence numbers per (batch, v-head), then eight 82432-byte
 * slots per (batch, v-head)).  Depends on the
 * kernel cgdr_prefill_path_for reports.  The workspace plays the part of the
 * single scratch arena of "Add parallel chunked prefill for channelwise gated
 * delta rule" (Summary), sliced per (batch, head) unit.  Returns 0 for
 * invalid arguments as well.
 */
size_t cgdr_prefill_workspace_size(const cgdr_args *args);

/*
 * Chunked prefill over T >= 0 tokens ("Add parallel chunked prefill for
 * channelwise gated delta rule", Summary): per chunk the per-channel
 * log-decay prefix, the causal query/key terms, the beta-folded triangular
 * (UT) transform, WY pseudo-keys and pseudo-values, and the inter-chunk
 * state carry, with a ragged last chunk handled by the same code.
 * T == 0 is a no-op.  The result equals T applications of the token
 * recurrence up to rounding, for every chunk length.
 * Paths: 1 <= T <= 8 runs the token recurrence itself (the decode kernel
 * stepping through the tokens, each state tile read once and written once;
 * the chunk length plays no part); otherwise bf16 inputs with dk = dv = 128
 * and chunk 64 run one of the three tensor-core kernels (tcgen05; TF32
 * operands for the anchored causal terms, fp16 operands for the other products
 * -- the per-head kernel keeps its state products in TF32 --, fp32
 * accumulation and state), and every other case an fp32
 * CUDA-core kernel; args->prefill_path can force a kernel for this call.
 * Workspace: the tensor-core path needs cgdr_prefill_workspace_size() bytes
 * (16-byte aligned); its first int32 is set to CGDR_ERR_TIMEOUT if a bounded
 * device wait gave up, or to CGDR_ERR_RANGE if an fp16 operand left the fp16
 * range (see cgdr_workspace_status).  `workspace` may be NULL
 * when the size is 0.  Returns CGDR_ERR_WORKSPACE if it is too small.
 */
cgdr_status cgdr_prefill(const cgdr_args *args, void *workspace, size_t workspace_bytes, void *stream);

/*
 * The kernels behind cgdr_prefill.  The three tensor-core kernels cover bf16
 * inputs with dk = dv = 128 and chunk 64 and agree up to rounding (the
 * cluster and cooperative kernels bit for bit); the CUDA-core kernel covers
 * every supported shape.  The split of the chunk's
 * work into a state-free part and the state carry follows the chunkwise form
 * of "Add parallel chunked prefill for channelwise gated delta rule"
 * (Summary); running them on different SMs has no counterpart there.
 */
typedef enum cgdr_prefill_path {
    CGDR_PREFILL_AUTO = 0,      /* per call: RECURRENT when 1 <= T <= 8; else COOP, CLUSTER or
                                   PER_HEAD, whichever needs the least time by the cycles per chunk
                                   each was measured at and how many heads each runs at once; SIMT
                                   for shapes the tensor-core kernels do not cover */
    CGDR_PREFILL_PER_HEAD = 1,  /* tensor cores, one CTA per (batch, v-head) */
    CGDR_PREFILL_CLUSTER = 2,   /* tensor cores, a cluster of four CTAs per (batch, v-head):
                                   one carries the state, three prepare chunks for it */
    CGDR_PREFILL_SIMT = 3,      /* fp32 CUDA cores, chunked */
    CGDR_PREFILL_RECURRENT = 4, /* 1 <= T <= 8: the token recurrence, fp32 CUDA cores, no
                                   workspace; for a longer T it means AUTO */
    CGDR_PREFILL_COOP = 5       /* tensor cores, one cooperative grid of one CTA per SM: a CTA per
                                   (batch, v-head) carries the state, every other CTA prepares
                                   chunks for all heads (needs more SMs than heads; else AUTO) */
} cgdr_prefill_path;

/*
 * The kernel cgdr_prefill would run for `args` on the current device, given
 * args->prefill_path: CGDR_PREFILL_PER_HEAD, CGDR_PREFILL_CLUSTER,
 * CGDR_PREFILL_COOP, CGDR_PREFILL_SIMT or CGDR_PREFILL_RECURRENT;
 * CGDR_PREFILL_AUTO (0) if `args` is invalid or there is nothing to do (B == 0
 * or T == 0).  A forced tensor-core kernel applies only to the shapes it covers
 * (else SIMT); COOP only with more resident CTAs than heads, and RECURRENT
 * only to 1 <= T <= 8 (else the automatic choice).  Queries the SM count, the
 * cluster capacity and the cooperative grid size once per device.
 */
int cgdr_prefill_path_for(const cgdr_args *args);

/*
 * Waits for `stream`, then reports the device-side status a cgdr_prefill
 * call left in `workspace`: CGDR_OK, CGDR_ERR_TIMEOUT if one of its bounded
 * waits on the tensor core gave up, or CGDR_ERR_RANGE if an fp16 operand left
 * the fp16 range (in both cases its outputs are invalid).
 * Returns CGDR_ERR_CUDA if the copy or the synchronisation fails.
 */
cgdr_status cgdr_workspace_status(const void *workspace, void *stream);

/*
 * Size, in bytes, of the library's static device scratch area used by
 * cgdr_prefill_noalloc.  Every GPU that loads the library holds this much
 * device memory until the process exits.
 */
#define CGDR_NOALLOC_SCRATCH_BYTES 4096

/*
 * cgdr_prefill without a caller-provided workspace, for callers that cannot
 * allocate device memory: runtimes that plan every device buffer ahead of
 * time and forbid allocation while a model runs, or code on a latency path
 * where a cudaMalloc (which may synchronise the device) is not acceptable.
 * This entry point has no counterpart in the method's description; it only
 * changes where the scratch memory comes from.
 *
 * The scratch lives in one file-scope static __device__ array of
 * CGDR_NOALLOC_SCRATCH_BYTES bytes.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.  The first call on
 * each device looks up that device's copy of the array (cudaGetSymbolAddress,
 * with the device current) and caches it; make that first call before any
 * stream capture.  Every call on a device shares the one array, which keeps
 * the last call's contents; the call clears what must start at zero before
 * its kernel runs.  Calls whose kernels overlap on the GPU (other streams,
 * other host threads) race on the array: serialise them.  A device-side
 * wait that gives up, or an fp16 operand out of range, is recorded in the
 * static area, which the caller cannot read, and in args->status when that
 * is given.
 *
 * Arguments and results are those of cgdr_prefill, except that a choice of
 * the cluster kernel (automatic or forced) runs the per-head tensor-core
 * kernel: the cluster kernel's hand-off ring does not fit the static area.
 * Returns CGDR_ERR_WORKSPACE if the problem needs more scratch than
 * CGDR_NOALLOC_SCRATCH_BYTES, and CGDR_ERR_CUDA if the set-up lookup fails.
 */
cgdr_status cgdr_prefill_noalloc(const cgdr_args *args, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CGDR_H_ */
