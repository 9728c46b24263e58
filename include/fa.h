/*
 * fa.h -- C ABI of libfa.so: exact, IO-aware fused attention on GB300
 * (sm_103a), forward and backward.
 *
 * The operation (the three-step form of "Reading CMU 11-868 LLM Systems:
 * FlashAttention", slide page 5, with a softmax scale and an optional causal
 * mask):
 *
 *     S = scale * Q K^T            (causal: S_ij = -inf for j > i)
 *     A = softmax(S) row by row
 *     O = A V
 *     lse_i = ln sum_j exp(S_ij)   (natural log, of the scaled scores)
 *
 * The forward kernel tiles Q by rows and streams K/V blocks through shared
 * memory with the online-softmax rescaling of cs2680 Lecture 9, sec. 9.4 and
 * the CMU post's slide page 12; only O and lse reach HBM.  The backward
 * kernels recompute S and P on chip from Q, K, V and lse (cs2680 Lecture 9,
 * sec. 9.6; CMU post, slide page 14) and never store an N x N matrix.
 *
 * Layout (all entry points): Q, K, V, O, dO, dQ, dK, dV are dense,
 * contiguous [B][H][N][d] arrays of bf16 (d innermost); lse and the
 * workspace's per-row terms are [B][H][N] fp32.  Causal masking is square
 * and top-left (row i attends to keys j <= i).
 *
 * Pointers: every tensor pointer is a DEVICE pointer of the current CUDA
 * device, 16-byte aligned, owned by the caller; the library neither frees
 * nor retains them past the call's stream work.  Outputs must not overlap
 * inputs (work items of one launch read inputs while others already write
 * outputs).  Calls are asynchronous on
 * `stream` (a cudaStream_t, NULL = legacy default stream) and never
 * synchronise, except fa_device_status().
 *
 * Errors: every entry point returns FA_OK (0) or a negative FA_ERR_* code.
 * On an argument error nothing is launched and no output is touched.  A
 * kernel whose internal pipeline wait exceeds its time limit stops early and
 * records FA_ERR_TIMEOUT in a per-device status word; fa_device_status()
 * reports it.
 *
 * Device state: the first call on a device caches, per device index, the
 * device addresses of the library's static device data (the status word,
 * the no-alloc scratch array, the forward pass's per-stream work counters)
 * and the SM count, and each stream that runs a masked forward pass keeps
 * its counter slot (see fa_fwd_schedule).  Do not use the library on a
 * device after cudaDeviceReset() in the same process: the cached addresses
 * belong to the context that the reset destroyed.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_ARG (-1)            /* null pointer, B/H/N < 1, non-finite scale, size overflow */
#define FA_ERR_UNSUPPORTED_D (-2)  /* head dimension d not in {64, 128} */
#define FA_ERR_ALIGN (-3)          /* a tensor pointer is not 16-byte aligned */
#define FA_ERR_WORKSPACE (-4)      /* workspace missing, misaligned or too small */
#define FA_ERR_DEVICE (-5)         /* current device is not sm_103 / no tcgen05, or no device */
#define FA_ERR_LAUNCH (-6)         /* a CUDA error was raised by a launch, or a
                                      kernel was compiled with fewer registers
                                      than its per-warpgroup register split
                                      needs (nothing is launched then) */
#define FA_ERR_TIMEOUT (-7)        /* a kernel's pipeline wait timed out (reported by fa_device_status) */
#define FA_ERR_BOUNDS (-8)         /* bounds-checked build only: a kernel computed a tile, mask
                                      or row index outside its array and stopped before using it
                                      (reported by fa_device_status) */

/*
 * Forward pass.
 *   q, k, v : [B][H][N][d] bf16, read only.
 *   o       : [B][H][N][d] bf16, written: O = softmax(scale Q K^T [+mask]) V,
 *             rounded to nearest-even from fp32.
 *   lse     : [B][H][N] fp32, written: ln sum_j exp(S_ij); the only
 *             per-row statistic kept for the backward pass.
 *   B, H, N : >= 1; d in {64, 128}; causal 0 or 1; scale finite (may be 0
 *             or negative).
 * Passes: cs2680 Lecture 9 sec. 9.4 (online softmax, running max m and
 * denominator l, correction by exp(m - m_new)); CMU post slide page 12.
 * Kernels: one CTA per work item by default.  With the environment
 * variable FA_FWD_PAIR=1 (read once per process), non-causal d = 128 calls
 * run on CTA pairs instead (tcgen05 cta_group::2, the 2-CTA products of the
 * CMU post's slide pages 50-52); both give bitwise the same results.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, int causal, float scale, void* stream);

/*
 * General forward pass: grouped query heads, N_q != N_kv, key splits.
 *   q, o   : [B][Hq][Nq][d] bf16 (o written); lse : [B][Hq][Nq] fp32 (written).
 *   k, v   : [B][Hkv][Nkv][d] bf16; Hq is a multiple of Hkv and query head h
 *            reads key/value head h / (Hq / Hkv) (GQA; MQA when Hkv = 1).
 *   causal : aligned bottom-right: query i sees keys j <= i + Nkv - Nq (the
 *            square top-left mask when Nq = Nkv); a query row that sees no
 *            key gets O = 0 and lse = -inf.
 *   num_splits >= 1: the keys are cut into that many ranges of whole
 *            128-key tiles (fewer if there are fewer tiles), processed in
 *            parallel and merged by their logsumexp -- the split-KV
 *            ("Flash-Decoding") scheme of cs2680 Lecture 9 sec. 9.8 and the
 *            CMU post's slide page 58, for short queries over long keys.
 *   workspace: with more than one effective split, a device buffer of at
 *            least fa_fwd_gqa_workspace_size(...) bytes, 256-byte aligned
 *            (per-split fp32 O and lse); otherwise it may be NULL.
 * The query heads of one key/value head are packed into the same 128-row
 * tiles (CMU post, slide page 59).  fa_fwd(...) is
 * fa_fwd_gqa(..., H, H, N, N, ..., 1, NULL, 0, stream).
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
               int Hkv, int Nq, int Nkv, int d, int causal, float scale, int num_splits,
               void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_gqa needs for these sizes and splits (0 when the
 * effective number of splits is 1 or the sizes are invalid). */
size_t fa_fwd_gqa_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int num_splits);

/* A number of key splits for these sizes on `sm_count` SMs: the smallest
 * split count, each split at least two 128-key tiles and at most 128 splits,
 * whose work items fill whole waves of SMs within 90% of the best count
 * (1 whenever the unsplit items already do).  Host only; negative FA_ERR_*
 * on bad arguments. */
int fa_fwd_gqa_splits(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal, int sm_count);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: an fp32 dQ
 * accumulator of B*H*ceil(N/128)*128*d floats, then two per-row fp32
 * terms of B*H*ceil(N/128)*128 floats each (-D_i with D_i = sum_k dO_ik
 * O_ik, and -lse_i * log2 e), each part rounded up to 256 bytes, then 256
 * bytes holding the main kernel's work-item counter.  Returns 0 when the
 * sizes are invalid.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass of fa_fwd, by recomputation.
 *   q, k, v, o, dout : [B][H][N][d] bf16, read only (o is fa_fwd's output).
 *   lse              : [B][H][N] fp32 from fa_fwd, read only.
 *   dq, dk, dv       : [B][H][N][d] bf16, written: the gradients of
 *                      L = sum(dout * O) with respect to q, k, v.
 *   workspace        : device buffer of at least
 *                      fa_bwd_workspace_size(B, H, N, d) bytes, 256-byte
 *                      aligned, owned by the caller; its contents on entry
 *                      do not matter and on return are unspecified.  Two
 *                      calls in flight at once need two workspaces.
 * dQ is accumulated in fp32 with atomic adds, so its last bits may differ
 * from run to run; dK and dV are deterministic.
 * Passes: cs2680 Lecture 9 sec. 9.6 (recompute the scores instead of
 * storing them); CMU post slide page 14 (the forward pass keeps only the
 * per-row normalisation constants).
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd split into its three kernels, for callers that want to time or
 * overlap them: bit 0 of phase_mask runs the preparation (-D_i and
 * -lse_i * log2 e, zeroing of the dQ accumulator and of the work-item
 * counter), bit 1 the main kernel (dK, dV and the dQ accumulation), bit 2
 * the dQ conversion to bf16.  fa_bwd(...) is fa_bwd_phases(..., 7).  Phases
 * must run in order on one stream with the same workspace, each main
 * kernel after its own preparation; arguments and errors as fa_bwd, plus
 * FA_ERR_ARG for a mask outside 1..7.
 */
int fa_bwd_phases(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, float scale, void* workspace, size_t workspace_bytes, void* stream,
                  int phase_mask);

/*
 * Block-sparse attention: the block-sparse extension of FlashAttention named
 * in the reading guide of cs2680 Lecture 9.  block_mask is a device array of
 * ceil(N/128) x ceil(N/128) bytes,
 * row-major, shared by every batch entry and head: key j is visible to query
 * i when block_mask[(i/128) * ceil(N/128) + j/128] is nonzero (and j <= i
 * when causal).  The 128 x 128 blocks are the kernels' own tiles, so a zero
 * entry skips that tile's loads and MMAs.  Masked scores count as -inf; a
 * query row with no visible key gets O = 0 and lse = -inf, and its rows of
 * the gradients are 0 (a key with no visible query gets dK = dV = 0).
 * All-ones masks give results bitwise equal to fa_fwd / fa_bwd.
 * Other arguments, ownership and errors as fa_fwd / fa_bwd, plus FA_ERR_ARG
 * for a null block_mask.  The mask must stay valid until the call's work on
 * the stream is done.
 */
int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, int causal, float scale, const void* block_mask,
                       void* stream);
int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, int causal, float scale, const void* block_mask,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 forward pass with incoherent processing (CMU 11-868 FlashAttention
 * post, FA3 section: FP8 as the low-precision direction, slide page 18, and
 * the Hadamard rotation of Q and K that spreads outliers, slide page 24).
 * Square shapes with d = 128 only (FA_ERR_UNSUPPORTED_D otherwise).
 *
 * Steps: with hadamard = 1 every row of Q and K is multiplied by the
 * 128 x 128 Sylvester Hadamard matrix H (entries +-1; (QH)(KH)^T = 128 QK^T);
 * each head of each of Q, K, V is quantised to E4M3 with one scale,
 * code = E4M3(x * (448 / amax)) rounded to nearest-even and saturated, amax =
 * max |x| over the head (amax = 0: codes 0, scale 1); then attention over the
 * codes: S = scale * (amax_q / 448)(amax_k / 448) * codes_q codes_k^T (/ 128
 * with the rotation), online softmax as in fa_fwd with P rounded to E4M3 as
 * the tensor-core operand of O += P V, O scaled by amax_v / 448.  O is bf16,
 * lse fp32 as in fa_fwd.
 *
 * Workspace (caller-owned, 256-byte aligned, fa_fwd_fp8_workspace_size
 * bytes), in this order with 256-byte aligned parts (offsets from
 * fa_fp8_workspace_offsets): q8 and k8, the codes of the (rotated) Q and K,
 * [B][H][N][128] bytes; vt8, the codes of V transposed per head,
 * [B][H][128][ceil(N/128)*128] bytes (keys past N hold code 0); amax,
 * [3][B][H] fp32 (Q, K, V, after the rotation).
 *
 * fa_fp8_quantize writes the workspace from bf16 q, k, v ([B][H][N][128]);
 * fa_fwd_fp8_quantized runs the attention kernel over a workspace written
 * by fa_fp8_quantize with the same sizes and hadamard flag; fa_fwd_fp8 is
 * the two in sequence on one stream.  Errors as fa_fwd, plus FA_ERR_ARG for
 * hadamard outside {0, 1}, FA_ERR_WORKSPACE for a missing, misaligned or
 * small workspace; fa_fp8_workspace_offsets fills offsets[4] (q8, k8, vt8,
 * amax) or returns an error; fa_fwd_fp8_workspace_size returns 0 for
 * invalid sizes.
 */
size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d);
int fa_fp8_workspace_offsets(int B, int H, int N, int d, size_t* offsets);
int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    int hadamard, void* workspace, size_t workspace_bytes, void* stream);
int fa_fwd_fp8_quantized(void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
                         int hadamard, const void* workspace, size_t workspace_bytes,
                         void* stream);
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, int causal, float scale, int hadamard, void* workspace,
               size_t workspace_bytes, void* stream);

/*
 * Size of the scratch array fa_bwd_noalloc uses: 32 MiB of static device
 * data on every GPU that loads the library, held until the process exits.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fa_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a deployment variant of fa_bwd, not part of the method.
 * Callers under a memory manager that owns all device memory, callers that
 * cannot afford cudaMalloc's implicit device-wide synchronisation, and
 * plugins given no allocator cannot provide fa_bwd's workspace; this entry
 * point takes it from a fixed scratch array in the library's static device
 * data instead and allocates nothing.
 *   Arguments, layouts and results as fa_bwd, without the workspace.
 *   Argument and alignment errors are checked first and returned as fa_bwd
 *   returns them; otherwise FA_ERR_WORKSPACE, launching nothing, when
 *   fa_bwd_workspace_size(B, H, N, d) > FA_NOALLOC_SCRATCH_BYTES (for
 *   d = 128 about 64K padded rows B*H*ceil(N/128)*128; for d = 64 about 127K).
 *   The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  All calls on a device share the one array
 *   and it keeps the previous call's contents (every part that is read is
 *   rewritten first): calls that overlap on the GPU race on it.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, void* stream);

/*
 * Synchronises `stream`, then returns and clears the status word of the
 * current device: FA_OK, FA_ERR_TIMEOUT if a kernel gave up on a pipeline
 * wait since the last call, FA_ERR_BOUNDS if a kernel of the bounds-checked
 * build caught an out-of-range index, or FA_ERR_LAUNCH if the stream holds a
 * CUDA error.  The first error recorded wins.  If `site` is not NULL it
 * receives the identifier of the wait or check that raised it (0 if none):
 * 101-199 a wait of the forward kernel, 201-299 one of the backward main
 * kernel, 1101-1199 a bounds check of the forward kernels, 1201-1299 one of
 * the backward kernels, FA_SITE_SELFTEST and FA_SITE_SELFTEST_BOUNDS the self
 * tests'.
 */
int fa_device_status(void* stream, int* site);

/*
 * Failure-detection self test (no counterpart on the pages): launches one
 * CTA whose thread waits, through the same bounded-wait path the kernels
 * use, on a shared-memory barrier that nothing completes.  After
 * timeout_us microseconds (1 .. 1000000) the wait gives up, records
 * FA_ERR_TIMEOUT with site FA_SITE_SELFTEST in the status word and the
 * kernel returns; the context stays usable.  Returns FA_ERR_ARG for a
 * timeout outside the range, else as a launch.
 */
#define FA_SITE_SELFTEST 901
int fa_selftest_timeout(int timeout_us, void* stream);

/*
 * Bounds-checked build (no counterpart on the pages).  Compiled with
 * FA_CHECKS defined, every kernel range-checks the tile, mask and row indices
 * it computes before it uses them; a violation records FA_ERR_BOUNDS and the
 * check's site in the status word, and the CTA winds down through the same
 * path as a timed-out wait (no trap, no access out of range).  The default
 * build compiles the checks out.  fa_checks_enabled() returns 1 in the
 * checked build and 0 otherwise.
 *
 * fa_selftest_bounds launches one thread that evaluates a bounds check on an
 * index one past its range, touching no memory but the status word: in the
 * checked build the status word then reads FA_ERR_BOUNDS at site
 * FA_SITE_SELFTEST_BOUNDS; in the default build it stays FA_OK.  Returns as
 * a launch.
 */
#define FA_SITE_SELFTEST_BOUNDS 902
int fa_checks_enabled(void);
int fa_selftest_bounds(void* stream);

/* A static, human-readable description of a status code. */
const char* fa_status_string(int status);

/*
 * The forward kernel's work list and its split over persistent CTAs.  A
 * work item is one (b*H + h, q-tile pair) unit: 256 query rows of one head.
 * Items are listed with heads in groups of 8 and, inside a group, longest
 * first (the LPT rule of the CMU post's slide pages 27-46: under a causal
 * mask later query tiles see more keys).  Without a mask the kernel runs
 * min(items, num_ctas) persistent CTAs (num_ctas = the device's SM count)
 * and CTA c takes the list in snake order (fa_snake_assign).  Under a causal
 * mask (and under a block mask) items differ in cost and are taken greedily
 * in list order (greedy list scheduling): with more items than num_ctas,
 * num_ctas persistent CTAs claim them from a device work counter as each
 * becomes ready for another, so item_cta is -1 (decided at run time);
 * otherwise item t gets CTA t.  The counter is the library's: one slot per
 * stream (streams told apart by handle; cudaStreamPerThread by host thread,
 * since it names a different stream in each), so launches on one stream
 * (which run in order) share it and launches on different streams do not; a
 * launch leaves its slot as it found it.  A CUDA graph that holds a masked forward pass uses the slot of
 * the stream it was captured on: it must not run at the same time as
 * another masked forward pass on that stream, nor twice at once.  After
 * 64 streams on a device have run masked forward passes, calls on further
 * streams give every item its own CTA instead (the hardware then hands CTAs
 * to SMs in list order as SMs free up).  Writes up to max_items entries of
 * item_bh, item_pair, item_cost (the item's number of 128-key tiles summed
 * over its two query tiles) and item_cta (any of them may be NULL) and
 * returns the number of items, or a negative FA_ERR_* code.  Host only;
 * needs no device.
 */
int fa_fwd_schedule(int B, int H, int N, int causal, int num_ctas, int* item_bh,
                    int* item_pair, int* item_cost, int* item_cta, int max_items);

/*
 * The static assignment of a list of n work items to `workers` persistent
 * workers used by the kernels: round k = i / workers of the list is dealt
 * to workers 0..workers-1 when k is even and in reverse when k is odd.  On
 * a longest-first list this balances the workers the way the LPT rule does
 * (the CMU post's example: costs 4,4,3,3,2,2,1,1 on 3 SMs give loads
 * 7,7,6).  Writes worker_of_item[0..n); returns FA_OK or FA_ERR_ARG.
 */
int fa_snake_assign(int n, int workers, int* worker_of_item);

/* Library version, for the loader's sanity check. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
