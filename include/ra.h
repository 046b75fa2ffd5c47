/*
 * ra.h -- C ABI of the blockwise exact attention library (libra.so), sm_103a.
 *
 * Exact softmax attention computed blockwise, as in "Ring Attention with
 * Blockwise Transformers for Near-Infinite Context" (arXiv 2310.01889,
 * Abstract: blockwise self-attention over key/value blocks that travel
 * around a ring of hosts, with no approximation).  On one GPU the ring is
 * emulated: P virtual hosts own contiguous row blocks of Q, K, V in device
 * memory and host i computes against key/value block (i - step) mod P at
 * each step ("Ring Attention: Train 1M Tokens on 8GB GPUs in 2026", section
 * "Ring Attention: Partition Sequence Length, Not Batch").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  q, k, v, o, dO, dq, dk, dv are [B, N, H, d] with d contiguous; by
 *   default packed with heads at stride d (the pages' [seq, heads, head_dim]
 *   layout with a batch axis; "Building Ring Attention in PyTorch: The
 *   200-Line Version"), and any batch, row and head strides through ra_shape
 *   (see there), so [B, H, N, d] tensors and slices of a fused projection
 *   need no copy.  Row blocks of a larger tensor are plain pointer offsets.
 *   The fp32 running state is o_acc [B, N_q, Hq, d] (packed) and m_acc,
 *   l_acc, lse [B, Hq, N_q] (packed).
 * Scores.  s_ij = scale * q_i . k_j; scale is usually d^-0.5 (same section).
 *   With RA_CAUSAL in `flags` key j is visible to query i iff
 *   kv_pos(j) <= q_pos(i), positions being global row indices (q_off /
 *   kv_off added for blocks).
 * State.  (m, l, o) is the triple the pages carry between ring steps
 *   (max_score, exp_sum, weighted_output; "Gotchas and Failure Modes"):
 *   l = sum_j exp(s_j - m), o = sum_j exp(s_j - m) v_j, m in natural-log
 *   units of the scaled scores.  m is a reference point, not necessarily
 *   the exact row maximum (kernels may defer rescaling while the maximum
 *   grows by less than 8 in log2 units); the represented quantities o/l and
 *   m + log(l) are what the state means.  A row that has seen no key has
 *   m = -inf, l = 0, o = 0.
 * Grouped heads.  Hq % Hkv == 0; query head h reads key/value head
 *   h / (Hq / Hkv).
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Every call only enqueues work and returns; it holds no pointer
 *   after it returns and allocates no device memory: the caller owns every
 *   buffer, including the workspace.  A call's work (kernels and the
 *   cudaMemsetAsync that zeroes its workspace's counters and accumulators)
 *   all goes to `stream`, so calls can be captured into a CUDA graph and
 *   replayed, provided one call has run on the device beforehand (the first
 *   call looks up the library's device status word).
 * Errors.  The return value reports argument validation and launch errors
 *   (ra_status).  Errors found on the device (a value out of fp16 range in a
 *   bf16 -> fp16 operand copy, a bounded wait that ran out) are recorded in a
 *   device status word; ra_sync_status() synchronises the stream and returns
 *   and clears it.  ra_last_error() gives a message for the last failure on
 *   the calling thread.
 * Precision.  RA_F32 inputs run in fp32 CUDA-core arithmetic (exact fp32
 *   products and sums).  RA_BF16 / RA_F16 inputs with d in {64, 128} run on
 *   the tcgen05 tensor cores with fp32 accumulation; the probabilities P
 *   (and dS in the backward pass) are rounded to fp16 for the second
 *   product, and bf16 operands of those products are copied to fp16 in the
 *   workspace first (exact for |x| in [2^-14, 65504]; larger values set
 *   RA_ERR_RANGE in the status word; smaller ones become fp16 subnormals,
 *   rounded to a multiple of 2^-24 without any status error).
 * Requirements.  Pointers 16-byte aligned; for ra_ring_fwd / ra_ring_bwd on
 *   tensor cores the host block N/P is a multiple of 128 rows; violations
 *   return RA_ERR_INVALID_ARG or RA_ERR_UNSUPPORTED.  Nothing falls back to
 *   another implementation.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { RA_F32 = 0, RA_BF16 = 1, RA_F16 = 2 } ra_dtype;

/* Bits of the `flags` argument.
 * RA_CAUSAL   key j is visible to query i only if kv_pos(j) <= q_pos(i).
 * RA_PRECISE  16-bit inputs: the operand rounded to fp16 for the second
 *             product (P in P V; dS in dS^T Q) is carried as two fp16 terms
 *             hi + lo, taking its rounding from 2^-12 to about 2^-24
 *             relative at the cost of one more MMA per tile.  Needed when
 *             logits are large and values have outliers (e.g. |q| ~ 4 N(0,1)
 *             with +-50 entries in V); ignored for RA_F32.
 * RA_STRIPED  ring entry points with RA_CAUSAL: the rows of q, k, v, o, dO,
 *             dq, dk, dv, lse are in striped order -- host i's local row l
 *             (tensor row i*S + l) holds sequence position l*P + i -- so every
 *             host has the same share of the causal triangle (load-balanced
 *             ordering; "Striped Attention" is named beside Ring Attention on
 *             "Ring Attention: Train 1M Tokens on 8GB GPUs in 2026", section
 *             "How Does This Compare to Other Long-Context Methods?").  The
 *             ring order is unchanged; every host visits every block, and in a
 *             (query host i, key host j) pair local key row lk is visible to
 *             local query row lq iff lk < lq, or lk == lq and j <= i.  In the
 *             backward pass a key tile's gradients go round the ring once per
 *             local query tile they meet (each lap in ring order), which keeps
 *             the query tiles that concurrent work units read in cache; only
 *             rounding depends on that order.  Ignored without RA_CAUSAL. */
enum { RA_CAUSAL = 1, RA_PRECISE = 2, RA_STRIPED = 4 };

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1, /* bad pointer, size, stride or alignment */
  RA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d = 96) */
  RA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  RA_ERR_RANGE = 4,       /* device: operand outside fp16 range */
  RA_ERR_TIMEOUT = 5      /* device: a bounded wait gave up */
} ra_status;

/* Sizes and strides.  The q group (q, o, dO, dq) and the kv group (k, v, dk,
 * dv) each share one layout: element (b, n, h, c) of a q-group tensor sits at
 * b * q_bstride + n * q_rstride + h * q_hstride + c (elements; d is always
 * contiguous), and likewise for the kv group.  A stride of 0 takes its packed
 * default: row stride H*d, head stride d, batch stride the extent of one
 * batch ((N-1)*rstride + (H-1)*hstride + d).  So zeroed strides describe the
 * pages' [seq, heads, head_dim] rows with a batch axis, and
 *   [B, H, N, d] tensors:  rstride = d, hstride = N*d, bstride = H*N*d;
 *   a slice of a fused [B, N, 3, H, d] projection: rstride = 3*H*d,
 *   hstride = d, bstride = N*3*H*d (outputs of the group need the same
 *   strides).
 * Strides must not make two (n, h) rows overlap, nor one batch overlap the
 * next; for 16-bit inputs on the tensor cores every stride is a multiple of 8
 * elements (16 bytes).  The fp32 running state o_acc/m_acc/l_acc and lse are
 * always packed.  Violations return RA_ERR_INVALID_ARG. */
typedef struct {
  int B;                /* batch */
  int N_q;              /* query rows covered by the call */
  int N_kv;             /* key/value rows covered by the call */
  int Hq;               /* query heads */
  int Hkv;              /* key/value heads (divides Hq) */
  int d;                /* head dimension */
  long long q_bstride;  /* elements between batches of q/o/dO/dq; 0 = packed */
  long long kv_bstride; /* elements between batches of k/v/dk/dv; 0 = packed */
  long long q_rstride;  /* elements between rows (positions) of q/o/dO/dq; 0 = Hq*d */
  long long q_hstride;  /* elements between heads of q/o/dO/dq; 0 = d */
  long long kv_rstride; /* elements between rows of k/v/dk/dv; 0 = Hkv*d */
  long long kv_hstride; /* elements between heads of k/v/dk/dv; 0 = d */
} ra_shape;

/* Set the running state to "nothing seen": o_acc = 0, m_acc = -inf,
 * l_acc = 0 (the ring loop's zero accumulators, "Building Ring Attention in
 * PyTorch: The 200-Line Version").  Uses shape.B, N_q, Hq, d. */
int ra_acc_init(float* o_acc, float* m_acc, float* l_acc, ra_shape shape,
                void* stream);

/* One ring step: fold the scores of a query block against one key/value
 * block into the running state (o_acc, m_acc, l_acc) with the online-softmax
 * rescale ("Gotchas and Failure Modes": keep (max, exp_sum,
 * weighted_output) and rescale on merge; online normaliser of Milakov and
 * Gimelshein cited by the arXiv 2310.01889 page).
 *   q      [B, N_q, Hq, d]  query block, global row position q_off + r
 *   k_blk, v_blk [B, N_kv, Hkv, d]  key/value block at positions kv_off + c
 *   dtype  type of q, k_blk, v_blk
 *   o_acc, m_acc, l_acc  state of the query block, read and updated
 *   flags  RA_CAUSAL / RA_PRECISE; key/value tiles wholly after a query
 *          tile are skipped, rows left with no visible key keep their state
 *   scale  score scale (> 0)
 *   workspace, ws_bytes  at least ra_block_fwd_workspace_bytes(dtype, shape)
 * Any N_q, N_kv >= 1 (ragged tiles are masked); tensor-core dtypes need
 * d in {64, 128}, RA_F32 d in {32, 64, 128}. */
int ra_block_fwd(const void* q, const void* k_blk, const void* v_blk,
                 ra_dtype dtype, float* o_acc, float* m_acc, float* l_acc,
                 ra_shape shape, long long q_off, long long kv_off, int flags,
                 float scale, void* workspace, size_t ws_bytes, void* stream);
size_t ra_block_fwd_workspace_bytes(ra_dtype dtype, ra_shape shape);

/* a <- merge(a, b) for two states of the same query rows: m = max(m_a, m_b),
 * l = l_a e^{m_a - m} + l_b e^{m_b - m}, o likewise; a side with m = -inf
 * has weight 0 ("Gotchas and Failure Modes").  Uses shape.B, N_q, Hq, d. */
int ra_merge(float* o_a, float* m_a, float* l_a, const float* o_b,
             const float* m_b, const float* l_b, ra_shape shape, void* stream);

/* Final normalisation of the state: O = o / l ("output / softmax_denom" at
 * the end of the ring loop) written as o_dtype, and lse = m + ln l (natural
 * log, saved for the backward pass).  Rows with l = 0 give O = 0 and
 * lse = -inf.  o_out has the q layout of `shape` (q_bstride honoured). */
int ra_finalize(const float* o_acc, const float* m_acc, const float* l_acc,
                void* o_out, ra_dtype o_dtype, float* lse, ra_shape shape,
                void* stream);

/* Whole forward ring in one call: P virtual hosts of S = N/P rows; host i
 * visits key/value blocks (i - s) mod P for s = 0..P-1, skipping blocks
 * wholly in its causal future, merges each block into its state and
 * normalises at the end ("Ring Attention: Partition Sequence Length, Not
 * Batch"; the loop of "Building Ring Attention in PyTorch: The 200-Line
 * Version" with the rescaled merge).
 *   q [B, N, Hq, d], k, v [B, N, Hkv, d] with N = shape.N_q = shape.N_kv
 *   o [B, N, Hq, d] in o_dtype; lse [B, Hq, N] fp32 (natural log)
 *   workspace: device memory, 256-byte aligned, at least
 *   ra_ring_fwd_workspace_bytes() bytes: for bf16/fp16 a 256-byte counter
 *   from which the kernel's CTAs draw their work (zeroed by each call), for
 *   bf16 also the fp16 copy of V; fp32 needs none (NULL allowed).  It must
 *   not be in use by work that overlaps the call on the GPU.
 * Tensor-core dtypes need S a multiple of 128. */
int ra_ring_fwd(const void* q, const void* k, const void* v, ra_dtype dtype,
                ra_shape shape, int P, int flags, float scale, void* o,
                ra_dtype o_dtype, float* lse, void* workspace, size_t ws_bytes,
                void* stream);
size_t ra_ring_fwd_workspace_bytes(ra_dtype dtype, ra_shape shape, int P);

/* Backward ring: gradients of L = sum(O * dO).  Probabilities are recomputed
 * from the saved lse (activation recomputation; "Building Ring Attention in
 * PyTorch" notes production code needs gradient checkpointing), and the
 * gradients of each key/value block travel with it around the ring: block
 * j visits hosts (j + s) mod P ("Gotchas and Failure Modes": gradients flow
 * backwards through the ring).
 *   D_i = dO_i . O_i; P_ij = exp(s_ij - lse_i); dV_j = sum_i P_ij dO_i;
 *   dS_ij = P_ij (dO_i . v_j - D_i); dQ_i = scale sum_j dS_ij k_j;
 *   dK_j = scale sum_i dS_ij q_i (summed over the query heads of a group).
 *   o in o_dtype, dO in dtype, lse from ra_ring_fwd; dq [B,N,Hq,d],
 *   dk, dv [B,N,Hkv,d] written in grad_dtype (fully overwritten).
 *   workspace: device memory, 256-byte aligned, at least
 *   ra_ring_bwd_workspace_bytes() bytes: D and LSE*log2(e) per row, for
 *   16-bit dtypes the fp32 dQ accumulator and the counter the kernel's CTAs
 *   draw their work from (both zeroed by each call), and for bf16 the fp16
 *   copies of q, k, v, dO.  It must not be in use by work that overlaps the
 *   call on the GPU. */
int ra_ring_bwd(const void* q, const void* k, const void* v, const void* o,
                ra_dtype o_dtype, const void* dO, const float* lse,
                ra_dtype dtype, ra_shape shape, int P, int flags, float scale,
                void* dq, void* dk, void* dv, ra_dtype grad_dtype,
                void* workspace, size_t ws_bytes, void* stream);
size_t ra_ring_bwd_workspace_bytes(ra_dtype dtype, ra_dtype grad_dtype,
                                   ra_shape shape, int P);

/* ra_ring_fwd for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is not available or not allowed (inside a host callback
 * or a custom allocator's own hooks, under a framework that owns every
 * device allocation, or with a fixed memory budget set at start-up) cannot
 * provide the workspace ra_ring_fwd asks for.  This entry point takes the
 * same arguments minus the workspace and uses a scratch buffer that is part
 * of the library itself: a device array of 32 MiB + 256 bytes per GPU that
 * loads the library, held until the process exits.  It allocates nothing.  The pages
 * describe no counterpart; it is a packaging of the same computation.
 *   Limit: shapes whose ra_ring_fwd_workspace_bytes() exceeds that size
 *   (the 256-byte work counter plus, for bf16 inputs, the fp16 copy of V,
 *   B*N*Hkv*d*2 bytes, at most 32 MiB) are rejected with RA_ERR_INVALID_ARG;
 *   fp16 inputs use only the counter, fp32 inputs no scratch.
 *   When the memory is taken: the array sits in a device module of its own
 *   (no kernel shares it).  Under CUDA's lazy module loading (the default
 *   since CUDA 12.2) a device reserves the 32 MiB at this entry point's
 *   first call there, when its address is looked up; with eager loading
 *   (CUDA_MODULE_LOADING=EAGER) every device the process creates a context
 *   on reserves them as soon as the library is loaded, whether or not this
 *   entry point is ever called.
 *   The first call on each device looks up the buffer's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   All calls share the one buffer per device and it keeps whatever the last
 *   call left there (each call zeroes the counter and overwrites the part it
 *   uses).  Calls whose work overlaps on the GPU (different streams,
 *   or threads without ordering between them) race on it. */
int ra_ring_fwd_noalloc(const void* q, const void* k, const void* v, ra_dtype dtype,
                        ra_shape shape, int P, int flags, float scale, void* o,
                        ra_dtype o_dtype, float* lse, void* stream);

/* Ring forward / backward with variable per-host lengths ("FAQ" of "Ring
 * Attention: Train 1M Tokens on 8GB GPUs in 2026": instead of computing on
 * padding, each host tracks which of its positions are valid and masks the
 * scores).  host_len is a device array of P int32: host i's first
 * host_len[i] rows (of S = N/P) hold its tokens, the rest is padding (values
 * are clamped to [0, S]).  The sequence is the valid rows in order, so a
 * causal mask keeps its block structure; padded keys are never visible,
 * padded query rows give O = 0, LSE = -inf, and padded rows get zero dQ, dK,
 * dV.  Key/value tiles or query tiles wholly in padding are skipped.  Other
 * arguments as in ra_ring_fwd / ra_ring_bwd; RA_STRIPED is not accepted. */
int ra_ring_fwd_varlen(const void* q, const void* k, const void* v, ra_dtype dtype,
                       ra_shape shape, int P, const int* host_len, int flags, float scale,
                       void* o, ra_dtype o_dtype, float* lse, void* workspace,
                       size_t ws_bytes, void* stream);
int ra_ring_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                       ra_dtype o_dtype, const void* dO, const float* lse, ra_dtype dtype,
                       ra_shape shape, int P, const int* host_len, int flags, float scale,
                       void* dq, void* dk, void* dv, ra_dtype grad_dtype, void* workspace,
                       size_t ws_bytes, void* stream);

/* One forward + backward step with the tensors in HOST memory: the work of
 * ra_ring_fwd followed by ra_ring_bwd, with the uploads and downloads it
 * needs.  The pages keep every block resident on its host and only move KV
 * between hosts; this call is for callers whose batches live in host memory
 * (a data loader, a CPU-side training loop).
 *   Inputs q, dO [B,N,Hq,d] and k, v [B,N,Hkv,d] in dtype; outputs o (o_dtype),
 *   lse [B,Hq,N] fp32 (packed), dq, dk, dv (grad_dtype); batch strides from
 *   `shape` apply to the host buffers.  All ten pointers are host pointers.
 *   workspace: device memory, 256-byte aligned, at least
 *   ra_ring_step_host_workspace_bytes() bytes; it holds the device copies and
 *   the forward and backward workspaces.
 *   Order: on `stream`, q, k, v go up, the forward runs, the backward runs,
 *   dq, dk, dv come down.  dO goes up on a library-owned side stream while the
 *   forward runs, and o and lse come down on a second one while the backward
 *   runs; both are joined back into `stream` with events, so the outputs are
 *   complete once `stream` has completed.  Pinned host memory (cudaHostAlloc,
 *   cudaHostRegister) makes every copy asynchronous; pageable memory works,
 *   but the copies then block the calling thread.  Two calls on two streams
 *   with two workspaces overlap one step's copies with the other's kernels.
 *   The workspace must not be in use by work that is not ordered before this
 *   call on `stream`.  The side streams are created on the first call on
 *   each device (make that call before any stream capture).
 *   Errors: everything ra_ring_fwd or ra_ring_bwd would reject is rejected
 *   before anything is enqueued; flags as for ra_ring_fwd. */
int ra_ring_step_host(const void* q, const void* k, const void* v, const void* dO,
                      ra_dtype dtype, ra_shape shape, int P, int flags, float scale,
                      void* o, ra_dtype o_dtype, float* lse, void* dq, void* dk, void* dv,
                      ra_dtype grad_dtype, void* workspace, size_t ws_bytes, void* stream);
size_t ra_ring_step_host_workspace_bytes(ra_dtype dtype, ra_dtype o_dtype,
                                         ra_dtype grad_dtype, ra_shape shape, int P);

/* Blockwise feed-forward layer ("Ring Attention with Blockwise Transformers
 * for Near-Infinite Context", Abstract: self-attention and the feedforward
 * network are both computed blockwise).  The layer is the Transformer's
 * position-wise feedforward
 *     y = GELU(x W1^T) W2^T,   GELU(u) = u Phi(u)  (exact, erf form),
 * computed one block of `block` tokens at a time so that only one block's
 * hidden activations [block, d_hidden] exist at once; the result is the same
 * as the unblocked layer.
 *   x, y [T, d_model] row-major (tokens of all batches); W1 [d_hidden, d_model],
 *   W2 [d_model, d_hidden] (output x input); x, W1, W2 (and dy) in `dtype`
 *   (RA_BF16 or RA_F16), y in y_dtype; fp32 accumulation on the tensor cores.
 *   Sizes: d_model and d_hidden multiples of 256, T and block multiples of 128
 *   (the last block may be shorter); else RA_ERR_UNSUPPORTED.
 *   workspace: device memory of ra_ffn_workspace_bytes() bytes (backward != 0
 *   for ra_ffn_bwd), 16-byte aligned; it holds the block's hidden activations.
 *   Ownership and errors as for ra_ring_fwd. */
size_t ra_ffn_workspace_bytes(ra_dtype dtype, long long T, int d_model, int d_hidden,
                              int block, int backward);
int ra_ffn_fwd(const void* x, const void* w1, const void* w2, ra_dtype dtype, long long T,
               int d_model, int d_hidden, int block, void* y, ra_dtype y_dtype,
               void* workspace, size_t ws_bytes, void* stream);

/* Backward of the blockwise feed-forward layer: gradients of L = sum(y * dy).
 * Each block recomputes its hidden activations h = x W1^T (no activation is
 * kept from the forward), then
 *     dH = (dy W2) * GELU'(h),  dx = dH W1,  dW2 += dy^T GELU(h),  dW1 += dH^T x.
 *   dx [T, d_model] in dx_dtype (fully overwritten); dw1 [d_hidden, d_model] and
 *   dw2 [d_model, d_hidden] fp32, zeroed by the call and summed over blocks.
 *   GELU(h), GELU'(h) and dH are rounded to `dtype` before they enter a
 *   product (they are tensor-core operands). */
int ra_ffn_bwd(const void* x, const void* w1, const void* w2, const void* dy, ra_dtype dtype,
               long long T, int d_model, int d_hidden, int block, void* dx, ra_dtype dx_dtype,
               float* dw1, float* dw2, void* workspace, size_t ws_bytes, void* stream);

/* Synchronise `stream`, then return and clear the device status word
 * (RA_OK, RA_ERR_RANGE or RA_ERR_TIMEOUT), or RA_ERR_CUDA if the stream
 * itself reports an error. */
int ra_sync_status(void* stream);

/* Message for the last non-OK return on the calling thread ("" if none). */
const char* ra_last_error(void);

/* Number of kernels this library has launched in this process. */
unsigned long long ra_launch_count(void);

/* Debug record of the ring schedule (off by default).  The pages debug a real
 * ring with one log file per rank that records what each step received
 * ("Ring Attention: Train 1M Tokens on 8GB GPUs in 2026", section "Debugging
 * Ring Transfers with Rank-Specific Logs"); here one process runs every
 * virtual host, and this log records, per tile the tensor-core kernels bring
 * into shared memory, which host's work it serves:
 *   entries  device array of `capacity` records of four uint32
 *            {kind, head, query tile, key tile}, 16-byte aligned:
 *            kind 0 -- the forward (ra_ring_fwd*, ra_block_fwd) loaded key/value
 *              tile `key tile` for the unit whose first query tile is
 *              `query tile` (128-row tiles, tensor row / 128);
 *            kind 1 -- the backward (ra_ring_bwd*) loaded query tile
 *              `query tile` for the unit of key/value tile `key tile`;
 *            head = b * Hq + (query head).
 *   count    device uint32 the kernels advance atomically (the caller zeroes
 *            it); records past `capacity` are counted but not stored.
 * One thread per CTA writes a unit's records, so they appear in the order the
 * unit visits its tiles (records of different units interleave).  Tiles that
 * are skipped (blocks in a query tile's causal future, tiles wholly in
 * padding) leave no record.  The setting is process-wide and applies to every
 * launch until ra_debug_visit_log(NULL, 0, NULL) turns it off; the buffers
 * must stay valid until then.  Logging costs one atomic per tile. */
int ra_debug_visit_log(unsigned int* entries, size_t capacity, unsigned int* count);

/* Kernel timing.  While enabled, every launch of the kernels below is
 * bracketed by CUDA events recorded on the stream it is launched on;
 * ra_kernel_timing_read() waits for those events and returns the summed
 * device time (ms) and the number of launches since timing was enabled.
 * ra_kernel_timing(1) enables and resets, ra_kernel_timing(0) disables and
 * releases the events.  Used by the benchmark to time the dominant kernel.
 * The two copy entries time ra_ring_step_host's transfers the same way: each
 * group of copies on one stream (q, k, v up; dO up; O and LSE down; dQ, dK,
 * dV down) is bracketed by events on that stream, so the sums are the time
 * the copies themselves took, whatever kernels ran beside them. */
typedef enum {
  RA_KERNEL_FWD_TC = 0,   /* tensor-core forward (ring and block step) */
  RA_KERNEL_BWD_TC = 1,   /* tensor-core backward */
  RA_KERNEL_FWD_F32 = 2,  /* fp32 CUDA-core forward */
  RA_KERNEL_BWD_F32 = 3,  /* fp32 CUDA-core backward (both kernels) */
  RA_KERNEL_GEMM_TC = 4,  /* tensor-core GEMM of the feed-forward layer (every launch) */
  RA_COPY_H2D = 5,        /* ra_ring_step_host uploads (two groups per call) */
  RA_COPY_D2H = 6,        /* ra_ring_step_host downloads (two groups per call) */
  RA_KERNEL_COUNT = 7
} ra_kernel_id;
int ra_kernel_timing(int enable);
int ra_kernel_timing_read(int kernel, double* total_ms, unsigned long long* launches);

/* Self-test of the bounded wait: launches one CTA that waits on an mbarrier
 * nobody arrives at, with a limit of timeout_us microseconds; the kernel must
 * give up, record RA_ERR_TIMEOUT in the status word and return.  Returns the
 * launch status; read the outcome with ra_sync_status(). */
int ra_selftest_timeout(unsigned int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
