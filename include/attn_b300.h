/*
 * attn_b300.h - C ABI of the exact IO-aware attention forward for B300 (sm_103a).
 *
 * The operation is the exact scaled-dot-product attention forward
 *
 *     O     = softmax(scale * Q K^T + causal mask) V
 *     LSE_i = ln sum_{j allowed for i} exp(scale * q_i . k_j)
 *
 * over the (batch, heads, seq_len, dim) problem statement of "Build a
 * FlashAttention kernel from scratch with Python and NumPy" (section
 * "Architecture Overview"), computed tile by tile with the online-softmax
 * update of "Building a FlashAttention-2 forward kernel in pure NumPy"
 * (sections "Architecture Overview" and "Step 3: Online softmax core") so
 * that the N x N score matrix never exists in memory.  The causal mask keeps
 * key j for query i when j <= i (the diagonal is kept, as the comment of the
 * first page's "Step 3" states).  LSE is the natural log of the sum of
 * exponentials of the scaled, masked scores: with the running max m and
 * running sum l of the FA-2 page's invariant, LSE = m + ln l.
 *
 * Layouts (all tensors row-major and contiguous, the contiguity that
 * "Flash Attention vs Standard Attention" asks of its inputs):
 *   dense  (cu_seqlens == NULL): q, k, v, o are (B, H, N, D); lse is (B, H, N).
 *   packed (cu_seqlens != NULL): the un-padded variable-length form of
 *          "Flash Attention vs Standard Attention" ("Critical Implementation
 *          Details"): B is the number of sequences and N the total token
 *          count; q, k, v, o are (H, N, D) and lse is (H, N).  cu_seqlens is
 *          a DEVICE int32 array of B+1 offsets; sequence s occupies tokens
 *          [cu_seqlens[s], cu_seqlens[s+1]).  Each sequence attends only to
 *          itself; causal positions are relative to the sequence start.
 *
 * Ownership and synchrony: every pointer is caller-owned device memory.  The
 * library allocates no device memory per call, keeps no pointer after a call
 * returns, and never synchronises the host: work is enqueued on `stream`
 * (a cudaStream_t; NULL means the legacy default stream) and the call
 * returns.  The host never reads cu_seqlens, so the grid is sized from N and
 * B and surplus CTAs exit at once.
 *
 * Work counters: the 16-bit forward (causal or packed) and the backward run
 * persistent CTAs that take their work items from a counter in the library's
 * static device memory (one of 256 per device, a new one per call, left at
 * zero by the last CTA of the launch).  Calls in flight at the same time get
 * different counters unless 256 of them are; the replays of one CUDA-graph
 * capture of a call reuse that call's counter, so they must not run
 * concurrently with each other (replays in stream order are fine).
 *
 * Errors: argument problems are reported synchronously by the return value
 * and nothing is launched.  Problems only the device can see (a wait that ran
 * out of time, cu_seqlens entries outside [0, N] or decreasing) set bits in a
 * per-device error word that attn_get_device_error() reads and clears; the
 * affected CTAs stop early and leave their outputs unwritten.  N == 0 is a
 * no-op that returns ATTN_OK.
 *
 * Thread safety: calls on distinct streams may come from distinct threads.
 */
#ifndef ATTN_B300_H
#define ATTN_B300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,     /* a required pointer is NULL (or only one of cu_seqlens_q/_k) */
  ATTN_ERR_SHAPE = -2,    /* B < 1, H < 1, N < 0, or sizes overflow the index types    */
  ATTN_ERR_HEADDIM = -3,  /* D not supported by this entry point                       */
  ATTN_ERR_ALIGN = -4,    /* q/k/v/o not 16-byte aligned, lse/cu_seqlens not 4-byte     */
  ATTN_ERR_ARCH = -5,     /* current device is not compute capability 10.3             */
  ATTN_ERR_LAUNCH = -6,   /* the CUDA runtime refused the launch or set-up              */
  ATTN_ERR_TIMEOUT = -7,  /* (device) a bounded wait inside a kernel ran out of time    */
  ATTN_ERR_BOUNDS = -8,   /* (device) cu_seqlens entries outside [0, N] or decreasing   */
  ATTN_ERR_SCALE = -9,    /* scale is not a finite number > 0                           */
  ATTN_ERR_SCRATCH = -10, /* attn_decode_noalloc: the problem needs more than the built-in
                             scratch (ATTN_NOALLOC_SCRATCH_BYTES); attn_bwd: the
                             workspace is smaller than attn_bwd_workspace_bytes()        */
  ATTN_ERR_DTYPE = -11    /* attn_fwd_cross: element type not one of attn_dtype          */
} attn_status;

/* Element type of q, k, v and o for attn_fwd_cross. */
typedef enum { ATTN_BF16 = 0, ATTN_F16 = 1, ATTN_F32 = 2 } attn_dtype;

/*
 * bf16 forward on tcgen05 tensor cores.
 *   q, k, v : const bf16 (__nv_bfloat16) device pointers, 16-byte aligned.
 *   o       : bf16 device output, same shape as q, 16-byte aligned.
 *   lse     : fp32 device output, natural log, 4-byte aligned.
 *   D       : 64 or 128.
 *   causal  : 0 or 1 (any non-zero value means 1).
 *   scale   : softmax scale (1/sqrt(D) in the usual case), finite and > 0.
 * Arithmetic: bf16 operands, fp32 accumulation of both products, fp32
 * softmax in base 2; the probabilities are rounded to bf16 for the second
 * product; O is rounded to bf16 once at the end.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int D, const int* cu_seqlens, int causal, float scale, void* stream);

/*
 * fp16 forward on tcgen05 tensor cores: the same as attn_fwd with IEEE
 * half-precision q, k, v and o (__half).  The probabilities are rounded to
 * fp16 for the second product and O is rounded to fp16 once at the end; the
 * rest of the arithmetic is as in attn_fwd.  This is the "mixed precision
 * fp16" variant named by "Build a FlashAttention kernel from scratch with
 * Python and NumPy" (section "Extending It", mixed-precision support).
 */
int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int D, const int* cu_seqlens, int causal, float scale, void* stream);

/*
 * fp32 forward on CUDA cores: same arguments and layouts with float tensors
 * (16-byte aligned), 1 <= D <= 128.  Scores, probabilities and accumulators
 * stay in fp32; exponentials use the accurate expf.
 */
int attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                 int H, int N, int D, const int* cu_seqlens, int causal, float scale,
                 void* stream);

/*
 * Forward with queries and keys of different lengths (cross-attention, which
 * "Python Attention Mechanisms Explained: From Self-Attention to Flash
 * Attention" names in section "The Core Idea").  The pages fix no mask for
 * this case; the causal mask here aligns the LAST query with the LAST key:
 * key j is allowed for query i when j <= i + (Nk - Nq).  With Nq < Nk the
 * queries are thus the last Nq positions of an Nk-long sequence and the
 * result equals the last Nq rows of causal self-attention over all Nk
 * positions; with Nq > Nk the first Nq - Nk queries see no key and get
 * O = 0, LSE = -inf.  Without the mask every query sees every key.
 *   dense  (cu_seqlens_q == cu_seqlens_k == NULL): q, o are (B, H, Nq, D),
 *          lse is (B, H, Nq); k, v are (B, H, Nk, D).
 *   packed (both non-NULL, DEVICE int32, B+1 entries each): q, o are
 *          (H, Nq, D) and lse (H, Nq) with Nq the total query tokens; k, v
 *          are (H, Nk, D) with Nk the total key tokens.  Sequence s has
 *          queries [cu_seqlens_q[s], cu_seqlens_q[s+1]) and keys
 *          [cu_seqlens_k[s], cu_seqlens_k[s+1]); the causal alignment is per
 *          sequence.  Passing only one of the two arrays is ATTN_ERR_NULL.
 *   dtype : ATTN_BF16 or ATTN_F16 (D in {64, 128}, tensor cores, the
 *          arithmetic of attn_fwd / attn_fwd_f16) or ATTN_F32 (1 <= D <= 128,
 *          the arithmetic of attn_fwd_f32).
 * Nk == 0 (or a sequence without keys) is allowed: those queries see no key,
 * and k, v may be NULL when Nk == 0.  attn_fwd, attn_fwd_f16 and attn_fwd_f32
 * are this call with Nk == Nq and cu_seqlens_k == cu_seqlens_q.  Device-side
 * checks, ownership and errors are as for attn_fwd.
 */
int attn_fwd_cross(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int Nq, int Nk, int D, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int causal, float scale, int dtype, void* stream);

/*
 * Forward from HOST buffers: attn_fwd_cross's dense self-attention (Nq = Nk =
 * N, no offsets) on q, k, v, o (B, H, N, D) and lse (B, H, N) that live in
 * host memory.  The planes are processed in up to 8 chunks through two
 * device slots in `workspace`; the copies to the device, the kernels and the
 * copies back of successive chunks run on three streams the library creates
 * once per device, so the two copy directions and the compute overlap.  The
 * host buffers must be page-locked (cudaHostAlloc / cudaHostRegister) for the
 * copies to overlap; pageable memory works but serialises them.  Work is
 * ordered after what `stream` already holds, and `stream` waits for the last
 * copy back: synchronise `stream` before reading o and lse.  Calls on one
 * device enqueue one at a time.  Argument checks and errors as for attn_fwd;
 * dtype as for attn_fwd_cross; a workspace smaller than
 * attn_fwd_host_workspace_bytes() returns ATTN_ERR_SCRATCH (it must be
 * 256-byte aligned).  This is the call a user with data in host memory makes;
 * the pages have no counterpart beyond their (batch, heads, seq_len, dim)
 * problem statement.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int D, int causal, float scale, int dtype, void* workspace,
                  unsigned long long workspace_bytes, void* stream);

/* Device workspace attn_fwd_host needs (two chunk slots); the size goes to *bytes. */
int attn_fwd_host_workspace_bytes(int B, int H, int N, int D, int dtype,
                                  unsigned long long* bytes);

/*
 * Backward pass: the gradients dQ, dK, dV of the forward for an upstream
 * gradient dO, with the probabilities rebuilt from the forward's saved
 * log-sum-exp -- the recomputation the "Building a FlashAttention-2 forward
 * kernel in pure NumPy" page names as the extension after the forward
 * ("Extending It: Your Roadmap to Senior-Level").  With P_ij =
 * exp(scale q_i.k_j - LSE_i) on the allowed keys (the mask of attn_fwd_cross):
 *     dV = P^T dO,  dS = P * (dO V^T - Delta),  Delta_i = dO_i . O_i,
 *     dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, B, H, Nq, Nk, D, cu_seqlens_q, cu_seqlens_k, causal, scale:
 *          as for attn_fwd_cross (the same layouts).
 *   o, lse : the forward's outputs for these inputs (o like q, lse fp32).
 *   dout   : dO, like q.          dq : like q.          dk, dv : like k.
 *   dtype  : ATTN_BF16 or ATTN_F16 (D in {64, 128}); ATTN_F32 is not offered.
 *   workspace : caller-owned device memory of attn_bwd_workspace_bytes()
 *          bytes, 16-byte aligned (Delta and an fp32 dQ accumulator); a
 *          smaller one returns ATTN_ERR_SCRATCH.
 * Arithmetic: 16-bit operands, fp32 accumulation of every product; P and dS
 * are rounded to the 16-bit type for the MMAs that take them; dQ is
 * accumulated over key tiles in fp32 and rounded once, as are dK and dV.
 * The order in which key tiles add into dQ is not fixed, so dQ may differ in
 * its last bits from run to run; dK and dV do not.
 * Packed layout: dk and dv rows outside every sequence are left untouched;
 * dq rows outside every sequence are written as 0.  Queries that see no key
 * get dQ = 0; keys that no query sees get dK = dV = 0.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int D,
             const int* cu_seqlens_q, const int* cu_seqlens_k, int causal, float scale, int dtype,
             void* workspace, unsigned long long workspace_bytes, void* stream);

/*
 * Workspace attn_bwd needs: packed != 0 for the packed layout (Nq is then the
 * total query tokens).  The size goes to *bytes.
 */
int attn_bwd_workspace_bytes(int B, int H, int Nq, int D, int packed, unsigned long long* bytes);

/*
 * KV-cache decode (bf16): Nq new query rows per (batch, head) attend to all Nk
 * cached keys, without a mask -- the incremental-decoding call of "Python
 * Attention Mechanisms Explained: From Self-Attention to Flash Attention"
 * (section "Causal Masking and Incremental Decoding"): a query of length 1
 * (here 1..8) against the key/value cache, is_causal=False.  Same definition of
 * O and LSE as attn_fwd with J(i) = every cached key.
 *   q : bf16 (B, H, Nq, D)        k, v : bf16 (B, H, Nk, D)
 *   o : bf16 (B, H, Nq, D)        lse  : fp32 (B, H, Nq)
 *   1 <= Nq <= 8, Nk >= 1, D in {64, 128}, scale finite and > 0.
 * The keys of each plane are split across thread blocks and the partial
 * results merged by their log-sum-exp.  The partials live in a caller-owned
 * device workspace of attn_decode_workspace_bytes() bytes (16-byte aligned);
 * with workspace == NULL (or too small) every plane is processed by one
 * thread block instead, which is correct but slower for few planes.
 * Arithmetic: bf16 operands, fp32 scores, sums and accumulators; the
 * probabilities are rounded to bf16 for P.V (as in attn_fwd), O is divided by
 * the sum of those rounded weights and LSE uses the fp32 sum; O is rounded to
 * bf16 once.
 */
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int D, float scale, void* workspace,
                unsigned long long workspace_bytes, void* stream);

/*
 * Workspace size attn_decode wants for this shape on the current device
 * (0 when one thread block per plane is already enough).  Returns a status;
 * the size goes to *bytes.
 */
int attn_decode_workspace_bytes(int B, int H, int Nq, int Nk, int D, unsigned long long* bytes);

/*
 * attn_decode_noalloc: attn_decode for callers that cannot allocate device
 * memory -- for example a host program embedded in another runtime that owns
 * every byte of device memory through its own pool (a cudaMalloc from here
 * would fail or fragment that pool), or latency-sensitive code that must not
 * pay for the device-wide synchronisation that freeing memory implies.  It
 * takes the same arguments as attn_decode except the workspace: the per-slice
 * partial results go to a scratch array built into the library, of
 * ATTN_NOALLOC_SCRATCH_BYTES per device, which every device that loads the
 * library holds until the process exits.  The call allocates nothing.
 *   - A problem whose partials need more than that returns ATTN_ERR_SCRATCH
 *     without launching (attn_decode_workspace_bytes gives the need).
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture.
 *   - Every call uses the same array and leaves its partials there; each call
 *     writes every entry it later reads, so nothing has to start at zero, but
 *     two calls that run on the GPU at the same time (different streams, or
 *     different host threads) overwrite each other's partials: keep them
 *     ordered, e.g. on one stream.
 * The attention pages have no counterpart to this entry point; it exists for
 * the callers above.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (2u << 20)
int attn_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int Nq, int Nk, int D, float scale, void* stream);

/* Static description of a status code. */
const char* attn_strerror(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (takes precedence) or
 * ATTN_ERR_BOUNDS; ATTN_ERR_LAUNCH if the synchronisation itself failed or a
 * kernel found its shared memory base misaligned and did not run.
 */
int attn_get_device_error(void* stream);

/*
 * Budget, in nanoseconds of GPU global time, of every bounded wait inside
 * the kernels launched after this call (default 1e9 = one second).  The
 * budget must exceed the longest wait a launch legitimately makes (a role
 * can wait for a whole query tile of another role, which grows with the
 * sequence length).  Returns ATTN_ERR_SHAPE below 1e6 (one millisecond).
 * A kernel whose wait ran out still waits for the copies and MMAs it has
 * already issued before it frees its tensor memory and exits; those drain
 * waits are bounded by the larger of this budget and one second, whatever
 * the budget.
 */
int attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * Abort-path test switch (on = 1, off = 0; anything else returns
 * ATTN_ERR_SHAPE).  While it is on, every launch of the forward, backward and
 * decode kernels makes its first thread block wait on an mbarrier phase
 * that nothing completes: that wait runs out of budget, the block raises its
 * abort flag, its other roles stop waiting, in-flight copies and MMAs
 * drain, tensor memory is freed and the block exits.  The call then reports
 * ATTN_ERR_TIMEOUT through attn_get_device_error, and its outputs are
 * undefined.  Nothing traps and the context stays usable.  It exists so that
 * tests can exercise the real kernels' timeout path; keep it off otherwise.
 * It applies to launches made after the call, from any thread.
 */
int attn_set_fault_injection(int on);

/*
 * Launches one CTA that waits on an mbarrier no thread ever arrives on, with
 * the given budget, through the same bounded-wait routine the attention
 * kernels use.  The wait gives up, records ATTN_ERR_TIMEOUT in the device
 * error word and the kernel returns; nothing traps and the context stays
 * usable.  Asynchronous like the other calls.
 */
int attn_wait_selftest(unsigned long long timeout_ns, void* stream);

/*
 * Measurement helper, not an attention operation (the pages have no
 * counterpart): reads `bytes` of device memory at `buf` once, as a
 * read-only stream (one block per SM copying 32 KB chunks into a 4-stage
 * shared-memory ring with 1-D TMA bulk copies), and XORs a fold of every
 * 32-bit word into the device word *out.  A bounded wait that runs out sets
 * ATTN_ERR_TIMEOUT in the device error word, as for the other kernels.  Timed
 * with CUDA events around it on `stream`, bytes / time is the read bandwidth
 * that bounds kernels which only read HBM (the KV-cache decode); a copy moves
 * twice the bytes and reaches a lower figure.  buf 16-byte aligned, bytes a
 * positive multiple of 16, out 4-byte aligned device memory (its prior value
 * is XORed into, not replaced).  Asynchronous; allocates nothing.
 */
int attn_hbm_read_probe(const void* buf, unsigned long long bytes, unsigned int* out,
                        void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_B300_H */
