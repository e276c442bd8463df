/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 forward library, libfa.so.
 *
 * Operation (one call = one forward pass over a whole batch):
 *   For every batch b, head h and query row i < Lq,
 *     S_ij  = scale * <Q[b,h,i,:], K[b,h,j,:]>           for allowed keys j
 *     O[b,h,i,:] = sum_j softmax_j(S_i.) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(S_ij)                      (natural log)
 *   Allowed keys: all j < Lk; with causal != 0 only j <= i (top-left aligned,
 *   diagonal kept).
 *
 * Where the operation is defined:
 *   - "Triton Ascend Attention" (skillmd.com), section 标准 Attention 计算流程:
 *     Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.
 *   - wsisp.com post "FlashAttention-2 forward in Triton": the host wrapper
 *     (Q, K, V of shape [B, H, L, D]; output O like Q; per-row statistic M of
 *     shape [B, H, Lq] in fp32; scale 1/sqrt(D)), the outer kernel's epilogue
 *     (M = m + log(l), O = O / l), and the inner loop (online softmax over
 *     streamed K/V tiles, causal mask offs_q >= offs_kv).
 *   - "flash-attention-kernel" skill card (skillsmp.com): head dims 64 and 128,
 *     causal keeps offs_m >= offs_n (diagonal included), tiles past the
 *     diagonal are skipped.
 *
 * Layout: Q [B,H,Lq,D], K and V [B,H,Lk,D], O [B,H,Lq,D], all bf16, contiguous,
 * row-major (D fastest).  LSE [B,H,Lq] fp32, contiguous.  All five pointers are
 * DEVICE pointers on the current CUDA device.
 *
 * Ownership: the caller allocates and owns every buffer.  The library keeps no
 * pointer after the call returns and allocates no device memory.  Q, K and V
 * are only read; O and LSE are only written and must not overlap Q, K, V or
 * each other.
 *
 * Execution: asynchronous on `stream` (0 = the legacy default stream).  The
 * call returns after the launch is queued.  Launch failures are reported by
 * the return value; failures detected by the kernel itself (a pipeline wait
 * that ran out of time) are reported by fa_last_device_status().
 */
#ifndef FA_H_
#define FA_H_

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O for fa_fwd_strided (LSE is always fp32). */
typedef enum {
    FA_DTYPE_BF16 = 0,
    FA_DTYPE_FP16 = 1
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* a null/misaligned/overlapping pointer, a bad size or scale */
    FA_ERR_UNSUPPORTED = 2,   /* D not in {64,128}, or the device is not sm_103 */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch, attributes, ...) */
    FA_ERR_TIMEOUT = 4        /* a kernel pipeline wait ran out of time (device status only) */
} fa_status;

/*
 * fa_fwd -- exact attention forward (the FlashAttention-2 forward pass).
 *
 *   Q, K, V : const bf16 device pointers, contiguous [B,H,Lq,D] / [B,H,Lk,D] / [B,H,Lk,D].
 *   O       : bf16 device pointer, [B,H,Lq,D], written (round to nearest even).
 *   LSE     : fp32 device pointer, [B,H,Lq], written: ln of the sum of exp of the
 *             scaled scores over the allowed keys of each row.
 *   B, H    : batch size and head count, >= 0.
 *   Lq, Lk  : query and key sequence lengths; Lq >= 0, Lk >= 1 (Lk = 0 would make
 *             every softmax empty).  Any lengths, not only multiples of 128.
 *   D       : head dimension, 64 or 128.
 *   causal  : 0 = every key; nonzero = key j allowed for row i iff j <= i.
 *   scale   : multiplies Q.K before the softmax; finite and > 0 (1/sqrt(D) is the
 *             usual choice).
 *   stream  : CUDA stream to launch on.
 *
 * Returns FA_OK once the kernel is queued.  B*H*Lq == 0 returns FA_OK without a
 * launch (pointers may then be NULL).  Argument errors return
 * FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED before anything is launched; all
 * pointers must be 16-byte aligned (the tensor-memory-access unit requires it).
 * Rows and keys are limited to 2^31-1 and B*H*L*D elements to 2^40.
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int Lq, int Lk, int D, int causal, float scale,
                 cudaStream_t stream);

/*
 * fa_fwd_workspace_size -- device workspace that fa_fwd_ws needs for this problem
 * on the current device, in *bytes (0: none).
 *
 * Same operation as fa_fwd, scheduled differently when few query tiles face long
 * key ranges.  Work is handed out in units of two 128-row query tiles of one head.
 * Causal units differ in cost and are balanced by ordering them heaviest first; when
 * the longest causal unit still takes at least twice an even share of all the key
 * tiles (a few heads of long sequences, units of at least 16 key tiles, at least two
 * key tiles per SM in all), its key range is cut as below.
 * Non-causal units all cost the same; when whole units would keep at most half of
 * the SMs busy in their last round and each unit has at least two 128-key tiles,
 * the key range of each unit is cut into consecutive pieces (the
 * FA-2 post's loop over K/V blocks, split between CTAs so every SM gets the same
 * number of key tiles).  Each piece leaves its rows' partial online-softmax state
 * (unnormalised O, running max m, exp-sum l -- the three per-row quantities of the
 * post's online-softmax section) in the workspace, and a second kernel on the same
 * stream merges them per row with the online-softmax update:
 *   m = max_k m_k,  O = sum_k 2^(m_k - m) O_k / sum_k 2^(m_k - m) l_k.
 * The workspace holds 2 x grid x 2 x 128 rows of (D + 2) floats (about 40 MB for
 * D = 128 on 152 SMs).
 * Returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED for arguments fa_fwd rejects on
 * sizes alone (and for bytes == NULL), FA_ERR_CUDA if the device cannot be queried.
 */
fa_status fa_fwd_workspace_size(int B, int H, int Lq, int Lk, int D, int causal, size_t* bytes);

/*
 * fa_fwd_ws -- fa_fwd with a caller-owned device workspace, which lets the
 * library use the split-key schedule above.  `workspace` must be 256-byte
 * aligned, hold at least the size fa_fwd_workspace_size reports and overlap no
 * other argument; it may be NULL when that size is 0.  Its contents on entry do
 * not matter; after the call it holds scratch.  Two calls that share a workspace
 * must not run concurrently.  When the split schedule is used, two kernels are
 * queued on `stream`.  Otherwise identical to fa_fwd (arguments, errors, results
 * up to the summation order of the merged rows).
 */
fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    int B, int H, int Lq, int Lk, int D, int causal, float scale,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Work schedules of the forward kernel, as fa_fwd_schedule reports them. */
typedef enum {
    FA_SCHED_WHOLE = 0,   /* whole units, heaviest first in a fixed order */
    FA_SCHED_SPLIT = 1,   /* key ranges cut across CTAs, merged by a second kernel */
    FA_SCHED_BAND = 2,    /* band-limited units (fa_fwd_window, key padding) */
    FA_SCHED_TABLE = 3    /* whole units in an order computed on the host */
} fa_schedule;

/*
 * fa_fwd_schedule -- the schedule fa_fwd_ws takes for this problem on the current
 * device, given a workspace of the size fa_fwd_workspace_size reports, in *schedule:
 *   FA_SCHED_SPLIT  when that size is nonzero (two kernels per call);
 *   FA_SCHED_TABLE  for causal problems whose heads' K and V take more than 48 MiB: the
 *                   host deals the units out head group by head group (about 32 MiB of
 *                   K/V per group, each unit to the least-loaded CTA), so a group's K/V
 *                   tiles stay in the L2 cache while its units run;
 *   FA_SCHED_WHOLE  otherwise.
 * The table and the fixed order give bit-identical results; the split schedule differs
 * only in the merge's summation order (see fa_fwd_ws).  fa_fwd (no workspace) takes the
 * same schedule except that it never splits.  Follows fa_debug_set (bit 4 turns the
 * table order off).  Errors as fa_fwd_workspace_size (schedule == NULL:
 * FA_ERR_INVALID_ARG); B*H*Lq == 0 gives FA_SCHED_WHOLE.
 */
fa_status fa_fwd_schedule(int B, int H, int Lq, int Lk, int D, int causal, int* schedule);

/*
 * fa_fwd_window -- local (sliding-window) attention: the operation of fa_fwd with
 * the allowed keys of row i restricted to a band around it,
 *     i - window_left <= j <= i + window_right   (and 0 <= j < Lk),
 * where -1 leaves that side unbounded.  Rows and keys are aligned at index 0 as
 * for the causal mask, which is the band (-1, 0); (-1, -1) is the full softmax.
 * The variant is the local / sliding-window attention that the wsisp.com post
 * "FlashAttention-2 forward in Triton" names among the masks FA-2 supports
 * (queries attend to a window of keys, not to all of them).  Key tiles outside
 * a query tile's band are skipped; only tiles the band's edges cut are masked.
 *
 *   window_left, window_right : >= -1.  A side at least Lq - 1 (left) or Lk - 1
 *     (right) keys wide covers every key on that side and counts as unbounded.
 *   Other arguments, layout, ownership and execution: as fa_fwd (whole units, no
 *   workspace; the bands (-1, 0) and (-1, -1) run fa_fwd's causal and full
 *   kernels).  LSE is taken over each row's band.
 *
 * Returns FA_ERR_INVALID_ARG for a side below -1, and when some row would have no
 * allowed key (window_left >= 0 and Lq - 1 - window_left > Lk - 1: the band of
 * the last row starts past the last key); otherwise as fa_fwd.
 */
fa_status fa_fwd_window(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        int B, int H, int Lq, int Lk, int D, int window_left, int window_right,
                        float scale, cudaStream_t stream);

/*
 * fa_fwd_strided -- the forward pass on strided tensors, in bf16 or fp16.
 *
 * The wsisp.com post "FlashAttention-2 forward in Triton" passes four strides per
 * tensor to its kernel (batch, head, row, feature) and stores O in fp16; this entry
 * point takes the first three of those strides (the feature stride is 1) for each of
 * Q, K, V and O, so layouts such as [B, L, H, D] or the Q/K/V parts of one packed
 * projection output are read in place, and it accepts fp16 as well as bf16.
 *
 *   Q, K, V  : const device pointers to elements of `dtype` (FA_DTYPE_BF16 or FA_DTYPE_FP16).
 *   q_stride, k_stride, v_stride, o_stride : host arrays of three element strides
 *              {batch, head, row}; element (b, h, i, d) of Q is at Q + b*s[0] + h*s[1] +
 *              i*s[2] + d.  Each stride of a dimension longer than 1 must be a
 *              non-negative multiple of 8 elements (16 bytes); Q, K and V may overlap
 *              (they are only read); no two elements of O may share an address, and O
 *              must not meet Q, K, V or LSE (checked on the byte spans the tensors cover).
 *   O        : device pointer, elements of `dtype`, written (round to nearest even).
 *   LSE      : fp32 device pointer, contiguous [B,H,Lq] (as fa_fwd).
 *   kv_len   : NULL, or a 4-byte aligned device array of B int32 key counts: key
 *              padding, another of the mask variants the post leaves to later work.
 *              Keys j >= kv_len[b] (clamped to [0, Lk]) are masked for every head and
 *              query of batch b, on top of the band.  The values are read by the kernel,
 *              so the host cannot see them: a row left with no allowed key (kv_len[b] = 0,
 *              or a band lying wholly in the padding) gets O = 0 and LSE = -inf instead
 *              of the argument error the band alone would give.  Key padding always runs
 *              the band schedule (never the split one).
 *   window_left, window_right : the band of fa_fwd_window; (-1, -1) is the full softmax
 *              and (-1, 0) the causal mask.
 *   workspace, workspace_bytes : optional (NULL, 0); with the full mask, a workspace of
 *              at least fa_fwd_workspace_size(B, H, Lq, Lk, D, 0) bytes lets the split
 *              schedule of fa_fwd_ws run.  A non-NULL workspace that is too small,
 *              misaligned or overlapping is an argument error.
 *   B, H, Lq, Lk, D, scale, stream : as fa_fwd.
 * Results are bit-identical to fa_fwd / fa_fwd_window / fa_fwd_ws on the same values
 * laid out contiguously (the addressing is the only difference).  Errors as those calls;
 * a bad stride or dtype is FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_strided(const void* Q, const long long* q_stride, const void* K,
                         const long long* k_stride, const void* V, const long long* v_stride,
                         void* O, const long long* o_stride, float* LSE, const int* kv_len,
                         int B, int H, int Lq, int Lk, int D, int window_left, int window_right,
                         float scale, int dtype, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * fa_fwd_noalloc -- fa_fwd_ws without a workspace argument, for callers that
 * cannot allocate device memory: code that only receives the input and output
 * pointers through a fixed interface with no allocator to ask, and code that
 * must not call cudaMalloc on its hot path because the call can synchronize the
 * device and take unbounded time.  The pages have no counterpart; this is a
 * packaging of the same computation.
 *
 * The split schedule's workspace lives in a 42 MiB device array inside this
 * library, reserved on every GPU that loads the library and held until the
 * process exits.  That covers the split schedule at D = 128 on GPUs with up to
 * 165 SMs (D = 64: 325 SMs); on larger GPUs a problem that would need more
 * returns FA_ERR_UNSUPPORTED before anything is launched.  Problems that run on
 * whole units (all causal ones, and non-causal ones that keep the SMs busy) use
 * no scratch at all.  Nothing is allocated by the call itself.
 *
 * The first call on each device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture.  The
 * address is kept for the life of the process: a cudaDeviceReset (or anything
 * else that destroys the device's primary context) makes it, like the library's
 * other per-device settings (among them the backward's stream and events), stale,
 * so after a reset no entry point of this
 * library may be called on that device again in the same process.  Every
 * call shares the one array and leaves scratch in it (it needs no clearing):
 * calls whose kernels can overlap on the GPU -- on different streams, or from
 * different host threads -- race on it and must be ordered by the caller.
 * Arguments, errors and results are otherwise those of fa_fwd_ws.
 */
fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                         int B, int H, int Lq, int Lk, int D, int causal, float scale,
                         cudaStream_t stream);

/*
 * fa_fwd_host_workspace_size -- device workspace that fa_fwd_host needs for this
 * problem on the current device, in *bytes (0 when B*H*Lq == 0): room for device
 * copies of Q, K, V, O and LSE (each rounded up to 256 bytes) followed by the split
 * schedule's workspace of the largest chunk that uses it (see fa_fwd_ws).
 * window_left / window_right as for fa_fwd_host.  Returns the argument errors of
 * fa_fwd_host that depend on sizes alone, FA_ERR_INVALID_ARG for bytes == NULL, and
 * FA_ERR_CUDA if the device cannot be queried.
 */
fa_status fa_fwd_host_workspace_size(int B, int H, int Lq, int Lk, int D, int window_left,
                                     int window_right, size_t* bytes);

/*
 * fa_fwd_host -- the forward pass on HOST buffers: Q, K, V are read from host memory,
 * O and LSE are written to host memory.  This is the host wrapper of the wsisp.com
 * post "FlashAttention-2 forward in Triton" (it takes the tensors, allocates O and
 * the per-row statistic M, runs the kernel and returns O) for callers whose tensors
 * live on the host, with the transfers made part of the call.
 *
 *   Q, K, V : host pointers, bf16, contiguous [B,H,Lq,D] / [B,H,Lk,D] / [B,H,Lk,D];
 *             only read.  Any alignment.
 *   O       : host pointer, bf16 [B,H,Lq,D], written;  LSE : host pointer, fp32
 *             [B,H,Lq], written.  O and LSE must not overlap Q, K, V or each other.
 *             Page-locked host memory (cudaHostAlloc / cudaHostRegister) lets the
 *             copies run asynchronously and overlap the kernels; pageable memory also
 *             works, with the copies then serialised by the CUDA runtime.
 *   window_left, window_right : the band of fa_fwd_window; (-1, -1) is the full
 *             softmax (fa_fwd with causal = 0, split schedule included) and (-1, 0)
 *             the causal mask (fa_fwd with causal != 0).
 *   workspace, workspace_bytes : DEVICE memory on the current device, 256-byte aligned,
 *             at least fa_fwd_host_workspace_size bytes, overlapping none of the host
 *             buffers; contents on entry do not matter, left as scratch (it holds the
 *             device copies of all five tensors).  Calls sharing a workspace must not
 *             run concurrently.
 *   B, H, Lq, Lk, D, scale : as fa_fwd.
 *   stream  : the call is ordered after the work already queued on `stream`, and
 *             `stream` completes only once O and LSE are in host memory.
 *
 * How it runs: the B*H (batch, head) slices are cut into up to 8 chunks of whole heads
 * (each large enough to keep the GPU busy); a long causal problem whose single head would
 * take the split-key schedule gets one more chunk, its last head alone, so that the
 * kernel left after the last upload is short.  Chunk c's Q, K, V travel to the device on
 * an internal upload stream while chunk c-1 is computed on `stream` (the kernels of
 * fa_fwd_ws / fa_fwd_window) and chunk c-2's O and LSE travel back on an internal
 * download stream; events order the three.  One cudaMemcpyAsync per tensor and chunk.
 * The call allocates no device memory; the two internal streams and their events are
 * created on the first call on each device and kept until the process exits.
 *
 * Asynchronous: the call returns once everything is queued; the host buffers must stay
 * valid and unmodified (Q, K, V) and unread (O, LSE) until `stream` has completed
 * (cudaStreamSynchronize).  Calls from several host threads are safe: each holds a
 * per-device lock while it queues its work.  B*H*Lq == 0 returns FA_OK with nothing
 * queued.  Argument errors are returned before anything is queued; FA_ERR_CUDA from a
 * failed copy or launch may leave part of the work queued (O and LSE are then
 * undefined).  Pipeline-wait timeouts are reported by fa_last_device_status().
 */
fa_status fa_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE,
                      int B, int H, int Lq, int Lk, int D, int window_left, int window_right,
                      float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_workspace_size -- device workspace fa_bwd needs, in *bytes: two fp32 arrays
 * (Delta_i = dO_i.O_i and LSE_i * log2(e)) over the query rows padded to whole
 * 128-row tiles, B*H*ceil(Lq/128)*128 entries each, each rounded up to 256 bytes, then
 * 256 bytes for the two kernels' work counters.  Argument errors as fa_bwd's
 * size checks (FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED; bytes == NULL is invalid).
 */
fa_status fa_bwd_workspace_size(int B, int H, int Lq, int Lk, int D, int causal, size_t* bytes);

/*
 * fa_bwd -- gradients of the attention of fa_fwd (the backward pass).
 *
 * Given the forward's inputs Q, K, V, its outputs O and LSE, and dO = dLoss/dO,
 * writes dQ, dK, dV = dLoss/dQ, dLoss/dK, dLoss/dV:
 *   P_ij  = exp(scale * Q_i.K_j - LSE_i)        (recomputed from LSE, not stored)
 *   dV_j  = sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i.V_j - Delta_i),  Delta_i = dO_i.O_i
 *   dQ_i  = scale sum_j dS_ij K_j,      dK_j = scale sum_i dS_ij Q_i
 * over the allowed pairs of the same mask as fa_fwd (causal: j <= i, top-left).
 * The wsisp.com post "FlashAttention-2 forward in Triton" states the principle
 * (recompute the probabilities from the saved row statistic instead of storing
 * them) and leaves the backward pass to later work; the formulas are the chain
 * rule through the forward definition.
 *
 *   Q, dO, O : const bf16 [B,H,Lq,D];  K, V : const bf16 [B,H,Lk,D];
 *   LSE      : const fp32 [B,H,Lq] as written by fa_fwd for the same arguments;
 *   dQ       : bf16 [B,H,Lq,D], written;  dK, dV : bf16 [B,H,Lk,D], written;
 *   workspace: device memory of at least fa_bwd_workspace_size bytes, 256-byte
 *              aligned, contents ignored and left as scratch (Delta, LSE*log2e and
 *              the counters from which the dK/dV and dQ kernels draw their work units);
 *   B, H, Lq, Lk, D, causal, scale, stream: as fa_fwd.
 * All pointers are device pointers, 16-byte aligned; dQ, dK, dV and the workspace
 * must not overlap each other or any input.  Three kernels are queued on `stream`
 * (Delta, then dK/dV, then dQ; dQ may start beside the last dK/dV units and
 * completes only after them, so stream order holds for whatever follows on
 * `stream`).  When B*H*ceil(Lk/128) (the dK/dV kernel's grid) is below the device's
 * SM count but that grid and the dQ kernel's, min(B*H*ceil(Lq/128), SMs), together
 * exceed it, the dQ kernel runs instead on a stream the library owns (one per device,
 * created by the first such call, with two events), beside the dK/dV kernel: that stream waits for the
 * Delta kernel through an event recorded on `stream`, and `stream` waits for the dQ
 * kernel through another, so stream order holds all the same.  A call that is being
 * captured into a CUDA graph takes the library's stream into the capture for its
 * duration (make a first such call before capturing, as it creates the stream); two
 * such captures on one device at once are not supported.  B*H*Lq == 0
 * with B*H*Lk > 0 zero-fills dK and dV;
 * B*H*Lk == 0 returns FA_OK with nothing queued.  Errors as fa_fwd; a pipeline
 * wait that runs out is reported by fa_last_device_status().
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Lq, int Lk,
                 int D, int causal, float scale, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/*
 * fa_bwd_masked -- fa_bwd under the band and key-padding mask of fa_fwd_strided: query
 * i attends to key j iff i - window_left <= j <= i + window_right (-1 = unbounded side)
 * and j < kv_len[b] (kv_len: NULL, or a 4-byte aligned device array of B int32 counts,
 * clamped to [0, Lk]).  LSE must come from the forward with the same mask (a row left
 * without keys has LSE = -inf there; it gets dQ = 0 and adds nothing to dK, dV).  The
 * bands (-1, -1) and (-1, 0) without kv_len are fa_bwd's full and causal masks.
 * Arguments, layout, workspace and errors otherwise as fa_bwd; a side below -1 or a
 * misaligned kv_len is FA_ERR_INVALID_ARG.
 */
fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                        const float* LSE, void* dQ, void* dK, void* dV, const int* kv_len, int B,
                        int H, int Lq, int Lk, int D, int window_left, int window_right,
                        float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_strided -- fa_bwd_masked on strided tensors, in bf16 or fp16: the backward
 * counterpart of fa_fwd_strided.  Each of Q, K, V, O, dO, dQ, dK, dV comes with three
 * element strides {batch, head, row} (features contiguous), under the rules of
 * fa_fwd_strided: 16-byte strides, no two elements of an output at one address, and
 * the outputs and the workspace meeting neither an input nor each other (inputs may
 * share memory).  dtype (FA_DTYPE_BF16 or FA_DTYPE_FP16) is the type of all eight
 * tensors; LSE stays fp32 [B,H,Lq] contiguous.  Results equal fa_bwd_masked's on the
 * same values laid out contiguously (bf16).
 */
fa_status fa_bwd_strided(const void* Q, const long long* q_stride, const void* K,
                         const long long* k_stride, const void* V, const long long* v_stride,
                         const void* O, const long long* o_stride, const void* dO,
                         const long long* do_stride, const float* LSE, void* dQ,
                         const long long* dq_stride, void* dK, const long long* dk_stride, void* dV,
                         const long long* dv_stride, const int* kv_len, int B, int H, int Lq,
                         int Lk, int D, int window_left, int window_right, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Human-readable name of a status code (static string; never NULL). */
const char* fa_status_string(fa_status s);

/*
 * fa_last_device_status -- synchronise `stream`, then read and clear the
 * library's device status words (forward and backward kernels) on the current device.  Returns FA_OK if no
 * kernel launched since the last read reported a problem, FA_ERR_TIMEOUT if a
 * pipeline wait inside a kernel gave up (the kernel then stops early and its
 * outputs are undefined), FA_ERR_UNSUPPORTED if a forward kernel found more work
 * units for one CTA than its shared-memory list holds (a planning error the host
 * is built to rule out; the CTA then computes nothing), or FA_ERR_CUDA if the
 * synchronisation failed.
 */
fa_status fa_last_device_status(cudaStream_t stream);

/*
 * fa_debug_set -- test hook, process-wide.  `wait_limit_ns` bounds every
 * pipeline wait inside the kernels (0 restores the default of one second).
 * `flags` bit 0 makes the load warp withhold the first value-tile load (of the
 * forward kernel, and of the backward's dK/dV kernel), so that the consumers' waits
 * run out and the kernel reports FA_ERR_TIMEOUT through fa_last_device_status()
 * instead of completing.  Bit 1 makes every
 * launch fail with FA_ERR_CUDA before anything is queued.  Bit 2 makes
 * fa_fwd_window run its band kernel also for the bands (-1, 0) and (-1, -1), so
 * that it can be compared with fa_fwd's kernels.  Bit 3 makes fa_fwd_host (and
 * fa_fwd_host_workspace_size) cut the heads into as many chunks as it can, so that
 * small problems exercise the overlapped pipeline.  Bit 4 turns off the host-computed
 * unit order that causal problems with more than 48 MiB of K/V use (heads grouped so
 * their K/V stay in the L2 cache, units dealt to the least-loaded CTA), so that the two
 * orders can be compared bit for bit.  Not for production use; returns FA_OK.
 */
fa_status fa_debug_set(unsigned int flags, unsigned long long wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
