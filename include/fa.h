/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact, IO-aware, tiled attention library.
 *
 * The library computes exact scaled-dot-product attention
 *     O = softmax(tau * Q K^T + mask) V
 * tile by tile with the online-softmax recurrence (running row max m, running
 * row sum l, accumulator rescaled by exp(m_old - m_new)), never writes the
 * N x N score or probability matrix to memory, and saves only O and the per-row
 * logsumexp.  The backward pass recomputes the probability tiles on chip from
 * Q, K, V and the logsumexp.  Sources of the method:
 *   - "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *     IO-Awareness" (Dao et al., 2022), as summarised on tonho.wtf (section
 *     "como funciona": the recurrence, the saved statistics, recomputation in
 *     the backward pass and D_i = dO_i . O_i) and agihunt.info (the fused
 *     forward/backward kernels, on-chip masking and dropout replay, and the
 *     block-sparse variant);
 *   - marketmaker.cc "Flash Attention" post (Q-outer loop, causal tile
 *     skipping, the PyTorch (batch, heads, seq, head_dim) interface);
 *   - lynx-cortex "FlashAttention como una optimizacion de roofline" (the
 *     Q-outer loop with deferred normalisation used by the forward kernel).
 *
 * Conventions shared by every entry point
 *   - Tensors Q, O, dO, dQ are logical [B, H, N, d] arrays of one dtype,
 *     addressed as base + b*stride_b + h*stride_h + n*stride_n + c (element
 *     strides; the head dimension is contiguous).  K, V, dK, dV are
 *     [B, H_kv, N, d] arrays of the same dtype with the kv_stride_* strides;
 *     H_kv = H (multi-head attention) unless grouped-query attention is asked
 *     for.  LSE is a contiguous float32 [B, H, N] array.
 *   - Grouped-query attention (living-dl-book, "Atencao eficiente", section
 *     6): the H query heads form H_kv groups of g = H / H_kv heads, and every
 *     head of group k reads K/V head k, i.e. query head h reads K/V head h / g;
 *     g = 1 is multi-head and g = H multi-query attention.  dK and dV of a
 *     shared head are the sums over its g query heads.
 *   - Sliding window (lynx-cortex, "Problemas de practica", the
 *     sliding-window exercise), read as the local causal window: with
 *     window = w > 0 and causal set, key j is visible to query i iff
 *     i - w < j <= i; whole K/V tiles outside every window of a query tile
 *     are skipped.
 *   - Head dimension: d = 64 for every dtype; d = 128 for float16 and
 *     bfloat16 (the pages name d = 128 as the case where the on-chip tile
 *     budget gets tight: marketmaker.cc, "O que isso custou"; lynx-cortex,
 *     "Lo que Flash forward no hace").  Other values, and d = 128 with
 *     float32, return FA_ERR_UNSUPPORTED.
 *   - Ownership: the caller owns every buffer and the stream.  The library
 *     never allocates, frees or synchronises device memory, except that
 *     fa_check_status synchronises the stream it is given.  Work is enqueued
 *     asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  All pointers named "device" must be device-accessible.
 *   - Errors found on the host (shapes, alignment, unsupported combinations,
 *     too small a workspace, a failed launch) are returned synchronously and
 *     nothing is enqueued.  There is no silent fallback to another algorithm:
 *     every unsupported combination returns FA_ERR_UNSUPPORTED.
 *   - Device-side waits are bounded; a wait that runs out records
 *     FA_ERR_TIMEOUT in the workspace status word, the kernel releases its
 *     resources and exits, and fa_check_status reports it.
 *   - Re-entrant: no global mutable state.  Concurrent calls need separate
 *     workspaces.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad probability ...   */
  FA_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement    */
  FA_ERR_MISALIGNED = 3,    /* base pointer or stride breaks the 16-B rule    */
  FA_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than the query says  */
  FA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed              */
  FA_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out             */
} fa_status;

typedef enum { FA_DT_F32 = 0, FA_DT_F16 = 1, FA_DT_BF16 = 2 } fa_dtype;

typedef struct {
  int32_t B, H, N, d;        /* batch, heads, sequence length, head dim         */
  int32_t dtype;             /* fa_dtype of Q,K,V,O,dO,dQ,dK,dV                 */
  int64_t stride_b;          /* element strides shared by all [B,H,N,d] tensors */
  int64_t stride_h;
  int64_t stride_n;
  float scale;               /* tau; <= 0 selects 1/sqrt(d)                     */
  int32_t causal;            /* nonzero: key j visible to query i iff j <= i    */
  const int32_t *seqlens_k;  /* device [B] or NULL: keys j >= L_b are masked     */
  float dropout_p;           /* in [0, 1); 0 disables dropout                   */
  uint64_t seed;             /* Philox4x32-10 key = (lo32(seed), hi32(seed))    */
  uint64_t offset;           /* Philox counter words 2,3 = (lo32, hi32)(offset) */
  const uint8_t *block_mask; /* device [nb][nb] (nb = ceil(N/block_size)),
                                nonzero = keep the block; or NULL (dense)       */
  int32_t block_size;        /* must be 128 when block_mask != NULL             */
  float *o_f32;              /* optional device [B,H,N,d] contiguous float32:
                                fa_fwd also writes O before its final rounding
                                to the storage dtype (parity diagnostics)       */
  void *prof_start;          /* optional cudaEvent_t pair: when both are set,   */
  void *prof_stop;           /* they are recorded on `stream` right before and
                                right after the main attention kernel of the
                                call (profiling; not owned by the library)      */
  /* -- ABI 1.1 -- zero-filled by callers of 1.0, which keeps their meaning */
  int32_t H_kv;              /* K/V heads; H % H_kv == 0; 0 selects H           */
  int64_t kv_stride_b;       /* element strides of K, V, dK, dV [B,H_kv,N,d];   */
  int64_t kv_stride_h;       /* all three 0 selects stride_b/h/n, allowed only  */
  int64_t kv_stride_n;       /* when H_kv == H                                  */
  int32_t window;            /* w > 0: key j visible to query i only if
                                i - w < j (requires causal); 0 = no window     */
  /* -- ABI 1.3 -- zero-filled by older callers, which keeps their meaning */
  int32_t fwd_kernel;        /* forward kernel at head dimension 64:
                                0 = chosen by the library (see fa_fwd);
                                1 = one 128-row query tile per CTA, two CTAs
                                    per SM; 2 = two query tiles per CTA
                                    sharing their K/V tiles.  Both compute
                                    the same result; other values and other
                                    head dimensions ignore it             */
} fa_params;

/* ---------------------------------------------------------------------------
 * fa_fwd_workspace_size / fa_bwd_workspace_size
 * Bytes of device workspace fa_fwd / fa_bwd need for `p` (0 is never
 * returned: the status word is always present).  Pure host function.
 * The backward workspace holds the float32 dQ accumulator [B,H,N,d] (16-bit
 * dtypes), D = rowsum(dO o O) [B,H,N], block lists and the status word.
 * ------------------------------------------------------------------------- */
size_t fa_fwd_workspace_size(const fa_params *p);
size_t fa_bwd_workspace_size(const fa_params *p);

/* ---------------------------------------------------------------------------
 * fa_fwd -- forward pass.
 * Computes, for every (b, h) head, O = P~ V with P = softmax(tau Q K^T) over
 * the visible keys (causal AND key-padding AND block mask), P~ = Z o P/(1-p)
 * when dropout is on, and LSE_i = m_i + ln l_i (natural log, tau-scaled
 * scores; -inf for a row with no visible key, whose O row is 0).
 * Method: Q-outer tiling with the online-softmax recurrence and deferred
 * normalisation (lynx-cortex, "El algoritmo Flash (forward)"; marketmaker.cc,
 * "O algoritmo de atencao do Flash"), whole future / masked / sparse tiles
 * skipped (marketmaker.cc, "O mascaramento causal"; agihunt.info, block-sparse
 * paragraph), dropout applied on chip (agihunt.info, fused-kernel paragraph).
 *   q, k, v : device [B,H,N,d] inputs (strides in p)
 *   o       : device [B,H,N,d] output, same dtype and strides
 *   lse     : device float32 [B,H,N] output
 *   ws      : device workspace of ws_bytes >= fa_fwd_workspace_size(p)
 * Dropout element (b,h,i,j) is kept iff the 16-bit slice (j & 7) of
 * Philox4x32-10(counter = (j>>3, (b*H+h)*N+i, lo32(offset), hi32(offset)),
 * key = (lo32(seed), hi32(seed))) is >= round(p * 65536); slice t is half
 * (t & 1) of output word (t >> 1), low half first.  Requires B*H*N < 2^32.
 * At head dimension 64 with fwd_kernel = 0 the library runs the one-tile
 * kernel unless the query tiles average at least 64 key tiles (dense or
 * causal, no window, no block mask) and the two-tile grid fills at least four
 * waves of the GPU, where sharing K/V tiles between two query tiles wins.
 * ------------------------------------------------------------------------- */
fa_status fa_fwd(const fa_params *p, const void *q, const void *k, const void *v,
                 void *o, float *lse, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * fa_bwd -- backward pass by recomputation (tonho.wtf, "como funciona": only
 * O, the softmax statistics and the RNG state are kept; S and P are rebuilt
 * on chip; D_i = dO_i . O_i replaces a length-N reduction).
 * For upstream gradient dO it computes, with the same mask and dropout
 * replay as fa_fwd:
 *   dV = P~^T dO;  dP = Z o (dO V^T)/(1-p);  D_i = dO_i . O_i;
 *   dS = P o (dP - D);  dQ = tau dS K;  dK = tau dS^T Q.
 *   q,k,v,o,dout : device [B,H,N,d] inputs;  lse: device float32 [B,H,N]
 *                  from fa_fwd with the same p
 *   dq,dk,dv     : device [B,H,N,d] outputs (same dtype and strides)
 *   ws           : device workspace, ws_bytes >= fa_bwd_workspace_size(p)
 * ------------------------------------------------------------------------- */
fa_status fa_bwd(const fa_params *p, const void *q, const void *k, const void *v,
                 const void *o, const void *dout, const float *lse,
                 void *dq, void *dk, void *dv, void *ws, size_t ws_bytes,
                 void *stream);

/* ---------------------------------------------------------------------------
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 * The FlashAttention pages have no counterpart; this is an interface
 * convenience around the same backward kernels.
 * Some callers cannot hand fa_bwd a workspace: code running inside a memory
 * pool it does not own, hooks where allocation is forbidden, or plain C
 * programs without a device allocator.  This entry point takes the
 * backward pass's scratch (dQ accumulator, padded LSE / D rows, status word)
 * from a fixed 64 MiB array compiled into the library's device image; every
 * device that loads the library holds that array until the process exits.
 * Arguments are those of fa_bwd without ws / ws_bytes.
 *   - Returns FA_ERR_WORKSPACE, enqueuing nothing, when
 *     fa_bwd_workspace_size(p) exceeds 64 MiB.  For 16-bit inputs the
 *     scratch is about 264 bytes per query row at d = 64 and 520 at
 *     d = 128 (float32 dQ accumulator, LSE and D), so B*H*N may reach about
 *     254,000 rows at d = 64 and 129,000 at d = 128; float32 inputs need
 *     8 bytes per row.  Block-sparse masks add their block lists.
 *   - The array's device address is looked up on every call (with the
 *     calling thread's current device).  The first call on a device also
 *     loads the library's device image there; make that first call before
 *     any stream capture.
 *   - All calls on a device share the array and leave their contents in it;
 *     what must start at zero is cleared on the stream by each call, but
 *     calls whose GPU work overlaps (unordered streams) race on it.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - A bounded device wait that gives up records FA_ERR_TIMEOUT in the
 *     array's status word: read it with fa_noalloc_check_status.
 * ------------------------------------------------------------------------- */
fa_status fa_bwd_noalloc(const fa_params *p, const void *q, const void *k, const void *v,
                         const void *o, const void *dout, const float *lse,
                         void *dq, void *dk, void *dv, void *stream);

/* fa_noalloc_check_status -- fa_check_status for fa_bwd_noalloc: synchronises
 * `stream`, then returns the status word the last fa_bwd_noalloc on the
 * current device left in the fixed array (FA_OK, or FA_ERR_TIMEOUT if a
 * bounded device wait ran out; the gradients are then undefined).
 * FA_ERR_CUDA if the stream reported an error. */
fa_status fa_noalloc_check_status(void *stream);

/* fa_noalloc_scratch -- the current device's address and size of the fixed
 * array fa_bwd_noalloc uses (for diagnostics: e.g. to run
 * fa_selftest_wait_timeout on it).  Allocates nothing. */
fa_status fa_noalloc_scratch(void **addr, size_t *bytes);

/* ---------------------------------------------------------------------------
 * fa_check_status -- synchronises `stream`, then reads the status word the
 * last fa_fwd/fa_bwd on `ws` left: FA_OK, or FA_ERR_TIMEOUT if a bounded
 * device wait ran out (outputs are then undefined).  FA_ERR_CUDA if the
 * stream reported an error.
 * ------------------------------------------------------------------------- */
fa_status fa_check_status(const void *ws, void *stream);

/* ---------------------------------------------------------------------------
 * fa_dropout_mask -- writes the dropout keep-mask fa_fwd/fa_bwd use for rows
 * row0 .. row0+nrows-1 of head (b, h): out[r][j] = 1 if kept, else 0, for
 * j in [0, N).  out: device uint8 [nrows][N].  Same mapping as fa_fwd.
 * For testing the mapping bit for bit; the attention kernels never store Z.
 * ------------------------------------------------------------------------- */
fa_status fa_dropout_mask(const fa_params *p, int32_t b, int32_t h, int32_t row0,
                          int32_t nrows, uint8_t *out, void *stream);

/* ---------------------------------------------------------------------------
 * fa_selftest_wait_timeout -- exercises the bounded device-side wait that
 * every attention kernel uses, without any attention work and without a
 * fault: one CTA of two warps waits on mbarriers that nothing arrives at,
 * the second warp starting one second after the first.  The first wait
 * gives up after the library's limit (2 s of %globaltimer), records
 * FA_ERR_TIMEOUT in the status word at the start of `ws` and raises the
 * CTA's abort flag; the second wait then returns on that flag, about one
 * second after it began.  The kernel exits normally and the context stays
 * usable.
 *   ws    : device workspace of >= 256 bytes (the status word is cleared
 *           first, as fa_fwd / fa_bwd do)
 *   out   : device int32[2]: 1 where a warp's wait returned "gave up"
 *   out_ns: device uint64[1]: nanoseconds the second warp waited
 * fa_check_status(ws) then returns FA_ERR_TIMEOUT.  For tests of the
 * failure path; it takes about two seconds.
 * ------------------------------------------------------------------------- */
fa_status fa_selftest_wait_timeout(void *ws, int32_t *out, uint64_t *out_ns, void *stream);

/* ---------------------------------------------------------------------------
 * FP8 forward (ABI 1.2).
 * FlashAttention-3's low-precision path (living-dl-book, "Atencao Eficiente
 * em Escala", section 10; marketmaker.cc, "FA3: Mecanica da tremonha", item
 * 3): Q, K and V are quantised to FP8 one tile at a time, with one scale per
 * tile, after a random Hadamard-style rotation of every row that spreads
 * outlying coordinates; the rotation is undone after the products.  Here:
 *   - FP8 is E4M3 (largest finite 448), round to nearest even, saturating;
 *   - the rotation is M = diag(signs) H_d / sqrt(d) (H_d the Sylvester
 *     Hadamard matrix); Q, K and V rows are all rotated; the scores are
 *     unchanged (M M^T = I) and O is rotated back, O = O' M^T;
 *   - a block is 128 rows x d of one head, scale = amax / 448, codes =
 *     E4M3(x * (448 / amax)); per_tensor = 1 uses the whole tensor's amax
 *     for every block and is the pages' baseline;
 *   - both products run in E4M3 on the tensor cores; the probabilities of
 *     key tile t are rounded to E4M3 as E4M3(exp(S - m) * 256 * sv_t / SV)
 *     with m the running row max (the accumulator is rescaled whenever m
 *     grows), sv_t the V scale of tile t and SV the largest V scale of the
 *     head; the row sum uses the unrounded probabilities;
 *   - head dimension 64 or 128, float16 or bfloat16 inputs and output; causal,
 *     key padding, block-sparse masks, the sliding window and grouped K/V
 *     heads as in fa_fwd; dropout returns FA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
typedef struct {
  int32_t per_tensor;        /* 0: one scale per 128-row block; 1: per tensor   */
  const int8_t *signs;       /* device int8 [d] of +1 / -1, 16-byte aligned:
                                rotate rows by diag(signs) H_d / sqrt(d);
                                NULL: no rotation                              */
} fa_fp8_params;

/* Byte offsets (multiples of 256) of the parts of the quantised buffer:
 *   q8  : uint8 [B,H,N,d]      E4M3 codes of the (rotated) Q rows
 *   k8  : uint8 [B,H_kv,N,d]   of K
 *   v8t : uint8 [B,H_kv,d,Np]  of V, transposed (keys contiguous), Np = N
 *                              rounded up to 128, zero on keys >= N
 *   sq  : float [B,H,nt]       dequantisation scale of each 128-row tile,
 *   sk, sv : float [B,H_kv,nt] nt = ceil(N / 128)
 *   amax: float [4]            scratch of the per-tensor mode
 * total is the buffer size. */
typedef struct {
  size_t q8, k8, v8t, sq, sk, sv, amax, total;
} fa_fp8_layout;

/* Fills *out for the problem p (a pure host function). */
fa_status fa_fp8_buffer_layout(const fa_params *p, fa_fp8_layout *out);

/* fa_fp8_quantize -- quantises q, k, v ([B,H,N,d] / [B,H_kv,N,d] 16-bit
 * tensors with the strides of p) into buf (device, 16-byte aligned,
 * buf_bytes >= layout.total).  The float32 order of operations is fixed:
 * sign flip, butterfly stages h = 1, 2, ..., d/2, multiply by 1/sqrt(d),
 * block amax, inv = 448 / amax, x * inv, E4M3 rounding. */
fa_status fa_fp8_quantize(const fa_params *p, const fa_fp8_params *f, const void *q, const void *k,
                          const void *v, void *buf, size_t buf_bytes, void *stream);

/* fa_fwd_fp8 -- the forward pass on a buffer fa_fp8_quantize filled with
 * the same p and f (f->signs rotates O back).  o: device [B,H,N,d] output in
 * p->dtype with p's strides; lse: device float32 [B,H,N] (natural log of
 * the scores of the dequantised operands); ws: ws_bytes >=
 * fa_fwd_workspace_size(p).  p->o_f32, if set, receives O before its final
 * rounding. */
fa_status fa_fwd_fp8(const fa_params *p, const fa_fp8_params *f, const void *buf, size_t buf_bytes,
                     void *o, float *lse, void *ws, size_t ws_bytes, void *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *fa_status_string(fa_status s);

/* Library ABI version (major * 100 + minor): 101 adds H_kv, kv_stride_*
 * and window to fa_params; 102 adds the FP8 forward; 103 adds fwd_kernel,
 * fa_noalloc_check_status and fa_noalloc_scratch. */
int32_t fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_FA_H */
