/*
 * uvu.h -- C ABI of the GB300 (sm_103a) channel-wise (UVU) Clebsch-Gordan tensor-product graph
 * convolution library (libuvu.so).
 *
 * The operation ("Receiver-streaming convolutions for channel-wise UVU tensor products",
 * OpenEquivariance discussion #221, opening post; "An Efficient Sparse Kernel Generator for
 * O(3)-Equivariant Deep Networks", abstract: CG tensor product fused with a graph convolution):
 *
 *   out[r,u,p,m3] = sum_{e : recv(e) = r} w[e,p,u] sum_{m1,m2} C^p[m1,m2,m3] x[src(e),u,l1,m1] Y[e,l2,m2]
 *
 * over the plan's paths p = (l1, l2, l3), and its vector-Jacobian product with respect to x, Y
 * and w.  C^p is the real Clebsch-Gordan tensor (unitary per output component, canonical sign:
 * the first non-zero entry in row-major (m1, m2, m3) order is positive; real basis with l = 1
 * ordered (y, z, x)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts (row-major, contiguous, one floating dtype per plan, indices int32):
 *     x      [N][U][D_x]      l1 blocks in irreps_x order
 *     Y      [E][D_Y]         l2 blocks in irreps_sh order (l*l + l + m for 0e+1o+2e+...)
 *     w, dw  [E][P][U]
 *     out, d_out [N][U][D_out]  path blocks in path order
 *     recv_offsets [N+1]      receiver CSR: edges of receiver r are [recv_offsets[r], recv_offsets[r+1])
 *     src    [E]              sender of each edge
 *     send_offsets [N+1], send_eids [E], send_recv [E]   transposed (sender) CSR
 * Path order: for each x irrep (string order), each SH irrep (string order), l3 ascending over
 * |l1-l2| .. min(l1+l2, lmax_out); every triangle-allowed l3 is kept, with parity p1*p2.
 *
 * Memory: every pointer is caller-owned DEVICE memory on the current device; floating-point
 * tensors are 16-byte aligned, int32 index arrays 4-byte aligned.  Because offsets are absolute
 * edge indices, a receiver sub-range [r0, r1) of a CSR is itself valid input: pass
 * recv_offsets + r0 with n_nodes = r1 - r0 and the matching rows of out / d_out (the edge-indexed
 * tensors keep their base pointers).  No entry point allocates device memory; the transpose takes a caller workspace.
 * Streams: work is enqueued on `stream` (0 = legacy default) and returns before it completes.
 * Once a plan's kernels for a call are loaded on the device (its first such call, which compiles
 * and loads the module), a call only enqueues kernel launches (and, for some, an asynchronous
 * memset) with no host synchronisation, so a sequence of calls can be recorded into a CUDA graph
 * by stream capture and replayed.
 * Outputs are overwritten, never accumulated: receivers without edges get out = 0, senders
 * without edges get dx = 0, n_edges == 0 writes zeros.
 * Errors: argument errors are detected on the host before anything is enqueued and return
 * UVU_ERR_INVALID_ARGUMENT; launch failures return UVU_ERR_CUDA; JIT failures return
 * UVU_ERR_COMPILE.  uvu_last_error_message() gives a per-thread description of the last error.
 * Graph contents (offsets monotone, indices in range) are trusted, not re-validated per call;
 * uvu_graph_validate() checks them on the device when asked.  No kernel traps, asserts or
 * waits on another kernel.
 */
#ifndef UVU_H_
#define UVU_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct uvu_plan_s *uvu_plan_t;
typedef struct CUstream_st *uvu_stream_t; /* same handle as cudaStream_t */

typedef enum { UVU_F32 = 0, UVU_F64 = 1 } uvu_dtype;

typedef enum {
    UVU_OK = 0,
    UVU_ERR_INVALID_ARGUMENT = 1,
    UVU_ERR_UNSUPPORTED = 2,
    UVU_ERR_COMPILE = 3,
    UVU_ERR_CUDA = 4,
    UVU_ERR_OUT_OF_MEMORY = 5
} uvu_status;

/* How dx is produced by uvu_conv_bwd. */
typedef enum {
    UVU_DX_SENDER = 0, /* sender-stationary over the transposed CSR, recomputing each edge's
                          contribution from w, Y and the gathered d_out row: no atomics,
                          deterministic, no workspace */
    UVU_DX_ATOMIC = 1, /* edge-parallel atomic scatter fused into the edge kernel (comparison);
                          summation order not deterministic */
    UVU_DX_STAGED = 2  /* the edge kernel writes each edge's dx contribution to a workspace, then a
                          sender-stationary kernel sums them over the transposed CSR in ascending
                          edge order: no atomics, deterministic, E*U*D_x*sizeof(dtype) bytes of
                          workspace */
} uvu_dx_mode;

/* ---------------------------------------------------------------------------- planning ---- */

/* Build a plan: parse the irreps, enumerate the paths, derive the real CG coefficients, emit
 * fully unrolled CUDA C++ with the CG non-zeros as immediates and compile it with NVRTC for
 * sm_103a.  Host only; the module is loaded on a device at its first launch there.
 * ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks", abstract: static
 * analysis at model compile time, long unrolled arithmetic instruction streams.)
 *   irreps_x   e.g. "128x0e+128x1o"; every term must share one multiplicity U (UVU); each l at
 *              most once; l <= 4.
 *   irreps_sh  e.g. "1x0e+1x1o+1x2e+1x3o"; every term multiplicity 1; l <= 4.
 *   lmax_out   0 <= lmax_out <= 8; bounds l3.
 *   plan_out   receives an opaque handle owned by the caller (free with uvu_plan_destroy).
 * Returns UVU_ERR_INVALID_ARGUMENT for a malformed string or a non-UVU multiplicity,
 * UVU_ERR_UNSUPPORTED for l beyond the limits or an empty path set, UVU_ERR_COMPILE when NVRTC
 * fails. */
uvu_status uvu_plan_create(const char *irreps_x, const char *irreps_sh, int lmax_out,
                           uvu_dtype dtype, uvu_plan_t *plan_out);

/* Release a plan and the modules it loaded.  NULL is accepted. */
uvu_status uvu_plan_destroy(uvu_plan_t plan);

/* Shapes of a plan.  Any output pointer may be NULL.  paths_l1l2l3, if not NULL, receives
 * 3*n_paths ints (l1, l2, l3 per path in path order). */
uvu_status uvu_plan_info(uvu_plan_t plan, int *mul_u, int *dim_x, int *dim_sh, int *dim_out,
                         int *n_paths, int *paths_l1l2l3);

/* The plan's real CG tensor of one path as fp64, dense (2l1+1)(2l2+1)(2l3+1), row-major in
 * (m1, m2, m3); `out` is caller-owned host memory of at least that many doubles. */
uvu_status uvu_plan_cg(uvu_plan_t plan, int path, double *out);

/* The emitted CUDA C++ source of the plan (valid until the plan is destroyed), and the NVRTC
 * log (ptxas resource usage).  Either pointer may be NULL. */
uvu_status uvu_plan_source(uvu_plan_t plan, const char **source, const char **compile_log);

/* A plan's generated modules: the convolution (forward, VJP; built by uvu_plan_create), and the
 * modules built on their first use: the double backward and the batched tensor product with
 * per-sample or batch-shared weights. */
typedef enum {
  UVU_MODULE_CONV = 0,
  UVU_MODULE_HVP = 1,
  UVU_MODULE_TP = 2,
  UVU_MODULE_TP_SHARED = 3
} uvu_module;

/* The emitted source and NVRTC log of one of the plan's modules.  Compiles it on the host if no
 * call has done so yet (no device needed); UVU_ERR_COMPILE if NVRTC fails,
 * UVU_ERR_INVALID_ARGUMENT for an unknown module.  The strings stay valid until the plan is
 * destroyed.  Either pointer may be NULL. */
uvu_status uvu_plan_module_source(uvu_plan_t plan, uvu_module module, const char **source,
                                  const char **compile_log);

/* Device-side status of the plan's kernels on the current device: bit 0 (UVU_DEV_TIMEOUT) is set
 * when a pipelined kernel, or a tensor-core product kernel (channel mixing, radial last layer;
 * their word is shared by all plans on the device), gave up waiting for a shared-memory stage or
 * for its matrix-multiply completion (about two seconds) and skipped the rest of its work, so
 * its outputs are not valid.  Synchronous: waits for all work
 * on the device, copies the word to *word and, if reset != 0, clears it.  Loads the plan's
 * module on the current device if needed. */
#define UVU_DEV_TIMEOUT 1u
uvu_status uvu_plan_device_status(uvu_plan_t plan, unsigned *word, int reset);

/* ------------------------------------------------------------------------- graph build ---- */

/* Receiver CSR from receiver-sorted edges ("Receiver-streaming convolutions ...", opening post,
 * benchmark paragraph: prepared, receiver-sorted edge lists; graph construction is not part of
 * the timed convolution).  recv_offsets[r] = #{e : recv[e] < r}.
 *   recv          device int32 [n_edges], non-decreasing, values in [0, n_nodes)
 *   recv_offsets  device int32 [n_nodes + 1], written
 * Bit-exact and deterministic.  A recv that breaks its precondition (a value outside [0, N) or
 * a decrease) gives an invalid CSR that uvu_graph_validate reports; no write leaves
 * recv_offsets. */
uvu_status uvu_csr_from_sorted_recv(int64_t n_nodes, int64_t n_edges, const int32_t *recv,
                                    int32_t *recv_offsets, uvu_stream_t stream);

/* Bytes of device workspace uvu_csr_transpose needs for these sizes. */
uvu_status uvu_csr_transpose_workspace(int64_t n_nodes, int64_t n_edges, size_t *bytes);

/* Transposed (sender) CSR: send_offsets [N+1]; send_eids [E] lists, per sender, the ids of
 * its edges in ascending edge-id order; send_recv[k] = receiver of edge send_eids[k].
 * Deterministic and bit-exact (the ordering is unique).  `workspace` is caller-owned device
 * memory of at least uvu_csr_transpose_workspace() bytes; its contents on entry do not matter.
 * Senders with up to 64 edges are ordered by rank counting, longer segments (hub senders) by an
 * in-place sort, O(d log^2 d) per segment of d edges. */
uvu_status uvu_csr_transpose(int64_t n_nodes, int64_t n_edges, const int32_t *recv_offsets,
                             const int32_t *src, int32_t *send_offsets, int32_t *send_eids,
                             int32_t *send_recv, void *workspace, size_t workspace_bytes,
                             uvu_stream_t stream);

/* Allocation-free variant of uvu_csr_transpose.  No counterpart in the paper: it exists for
 * callers that cannot provide device memory of their own, such as a plugin whose host runtime
 * owns the whole device memory pool and passes it only input and output buffers, or a
 * latency-critical path that must not take an allocator lock or risk running out of memory in
 * the middle of its work.  Same arguments and results as uvu_csr_transpose, without the
 * workspace: the scratch is a fixed 16 MiB array compiled into the library, present on every
 * GPU that loads it until the process exits.  Graphs needing more than that
 * (uvu_csr_transpose_workspace() > 16 MiB, i.e. roughly 4(N+1) + 4E > 16 MiB) are rejected with
 * UVU_ERR_UNSUPPORTED before anything is enqueued.  This function allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library call).  Each call made outside stream capture
 * looks up the array's device address on the current device (cudaGetSymbolAddress; the first
 * such call on a device also loads the array there), so a device reset in between leaves no
 * stale address.  A call on a capturing stream reuses the address found by the last call on that
 * device: make one call on each device before any stream capture (a capture before it returns
 * UVU_ERR_INVALID_ARGUMENT).  Every call re-initialises the scratch it reads, so the previous
 * call's leftovers do not matter, but all calls share one array: calls whose work overlaps on the
 * GPU race. */
uvu_status uvu_csr_transpose_noalloc(int64_t n_nodes, int64_t n_edges, const int32_t *recv_offsets,
                                     const int32_t *src, int32_t *send_offsets, int32_t *send_eids,
                                     int32_t *send_recv, uvu_stream_t stream);

/* Check a receiver CSR and sender list on the device: offsets[0] == 0, non-decreasing,
 * offsets[N] == E, 0 <= src < N.  Synchronises `stream`; *n_bad receives the number of
 * violations (0 = valid).  `workspace` needs 8 bytes of device memory. */
uvu_status uvu_graph_validate(int64_t n_nodes, int64_t n_edges, const int32_t *recv_offsets,
                              const int32_t *src, void *workspace, int64_t *n_bad,
                              uvu_stream_t stream);

/* ------------------------------------------------------------------------ convolution ---- */

/* Forward, receiver-stationary streaming: each (receiver, channel) owner scans its receiver's
 * edges and reduces in registers; no per-edge intermediate touches global memory
 * ("Receiver-streaming convolutions ...", opening post, ownership paragraph).  out is
 * overwritten.  One kernel launch. */
uvu_status uvu_conv_fwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                        const void *Y, const void *w, const int32_t *recv_offsets,
                        const int32_t *src, void *out, uvu_stream_t stream);

/* Backward edge kernel: per edge, channels in parallel; writes dw directly and reduces dY
 * across channels inside the block, with no atomics ("Receiver-streaming convolutions ...",
 * opening post, backward paragraph).  dY and dw are overwritten; either may be NULL (skipped).
 * If dx_atomic is not NULL, dx is first zeroed and then accumulated by atomic adds from the
 * same kernel (the atomic-scatter variant; its summation order is not deterministic).
 * If dx_edge is not NULL (device [E][U][D_x]), each edge's dx contribution
 * sum_p w[e,p,u] sum_{m2,m3} C Y[e] d_out[recv(e)] is written there, to be summed per sender by
 * uvu_conv_bwd_dx_reduce (UVU_ERR_UNSUPPORTED for a plan whose kernels cannot produce it).
 * One kernel launch (plus a memset when dx_atomic is given). */
uvu_status uvu_conv_bwd_edge(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                             const void *Y, const void *w, const int32_t *recv_offsets,
                             const int32_t *src, const void *d_out, void *dY, void *dw,
                             void *dx_atomic, void *dx_edge, uvu_stream_t stream);

/* Sender-stationary reduction of per-edge dx contributions: dx[s,u,:] = sum over the sender's
 * edges (transposed CSR, ascending edge id) of dx_edge[e,u,:].  Written once per sender, no
 * atomics, bitwise deterministic ("Receiver-streaming convolutions ...", reply on source- vs
 * destination-stationary convolutions: the dx side owned by the source node).
 * One kernel launch. */
uvu_status uvu_conv_bwd_dx_reduce(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges,
                                  const int32_t *send_offsets, const int32_t *send_eids,
                                  const void *dx_edge, void *dx, uvu_stream_t stream);

/* Bytes of device workspace uvu_conv_bwd needs in dx_mode (0 except for UVU_DX_STAGED). */
uvu_status uvu_conv_bwd_workspace(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges,
                                  uvu_dx_mode dx_mode, size_t *bytes);

/* Backward dx, sender-stationary: each (sender, channel) owner walks the sender's edges through
 * the transposed CSR and writes dx once, without atomics; deterministic (bitwise repeatable)
 * ("Receiver-streaming convolutions ...", source- vs destination-stationary reply).
 * One kernel launch. */
uvu_status uvu_conv_bwd_dx(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *Y,
                           const void *w, const int32_t *send_offsets, const int32_t *send_eids,
                           const int32_t *send_recv, const void *d_out, void *dx,
                           uvu_stream_t stream);

/* Full VJP: dx, dY, dw (any may be NULL = not computed).  dx_mode selects how dx is formed; the
 * transposed-CSR arguments may be NULL when dx_mode == UVU_DX_ATOMIC or dx == NULL, and
 * send_recv may be NULL for UVU_DX_STAGED.  `workspace` (caller-owned device memory of at least
 * uvu_conv_bwd_workspace() bytes, 16-byte aligned) is needed by UVU_DX_STAGED only.
 * Launches: SENDER 2 kernels, ATOMIC 1 kernel + 1 memset, STAGED 2 kernels. */
uvu_status uvu_conv_bwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                        const void *Y, const void *w, const int32_t *recv_offsets,
                        const int32_t *src, const int32_t *send_offsets,
                        const int32_t *send_eids, const int32_t *send_recv, const void *d_out,
                        void *dx, void *dY, void *dw, uvu_dx_mode dx_mode, void *workspace,
                        size_t workspace_bytes, uvu_stream_t stream);

/* Double backward (Hessian-vector product) of the convolution, for force training
 * ("Receiver-streaming convolutions ...", results table: HVP column; "An Efficient Sparse Kernel
 * Generator ...", abstract: higher partial derivatives for interatomic forces).  Given the
 * cotangents ax [N][U][D_x], aY [E][D_Y], aw [E][P][U] of the VJP outputs (dx, dY, dw) for the
 * cotangent d_out, it returns the gradients of
 *     L2 = <ax, dx> + <aY, dY> + <aw, dw>
 * with respect to d_out, x, Y and w.  Because the output is linear in each of x, Y, w, these
 * are forward and VJP contractions with one argument substituted:
 *     grad_d_out = F(ax,Y,w) + F(x,aY,w) + F(x,Y,aw)      [N][U][D_out]
 *     grad_x     = dx(Y<-aY) + dx(w<-aw)                  [N][U][D_x]
 *     grad_Y     = dY(x<-ax) + dY(w<-aw)                  [E][D_Y]
 *     grad_w     = dw(x<-ax) + dw(Y<-aY)                  [E][P][U]
 * A NULL cotangent counts as zero; a NULL output is not computed.  grad_x is formed from
 * per-edge contributions summed per sender over the transposed CSR (deterministic) when
 * uvu_conv_hvp_workspace() reports a non-zero size, which needs that much caller workspace;
 * otherwise (direct-load plans, U < 32, with several register groups) by atomic adds into a
 * zeroed grad_x.  The plan's HVP kernels are compiled on its first HVP call (host, NVRTC) and
 * loaded once per device; for U >= 32 they are the bulk-copy pipelined kernels of the forward
 * and edge backward with the cotangent rows in the same stages, and their bounded waits report
 * through uvu_plan_device_status like the plan's other kernels.
 * Launches: uvu_hvp_fwd (if grad_d_out), uvu_hvp_edge (if grad_x, grad_Y or grad_w), and the
 * sender-stationary reduction for grad_x. */
uvu_status uvu_conv_hvp(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                        const void *Y, const void *w, const int32_t *recv_offsets,
                        const int32_t *src, const int32_t *send_offsets, const int32_t *send_eids,
                        const void *d_out, const void *ax, const void *aY, const void *aw,
                        void *grad_d_out, void *grad_x, void *grad_Y, void *grad_w,
                        void *workspace, size_t workspace_bytes, uvu_stream_t stream);

/* Bytes of device workspace uvu_conv_hvp needs for grad_x (0 when it uses atomic adds). */
uvu_status uvu_conv_hvp_workspace(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, size_t *bytes);

/* ------------------------------------------- receiver- vs sender-stationary forward ---- */

/* The two ownerships of the convolution's forward ("Receiver-streaming convolutions ...",
 * replies: a source-stationary and a destination-stationary convolution behind one interface,
 * the one that moves less data determined from the irreps at init time; opening post: a mode
 * argument selects an implementation, the auto mode picks one). */
typedef enum { UVU_FWD_AUTO = 0, UVU_FWD_RECEIVER = 1, UVU_FWD_SENDER = 2 } uvu_fwd_mode;

/* Data-movement model of the two forwards for a graph of this size: bytes moved per launch by
 * the receiver-stationary forward (w, Y, one gathered x row per edge, one out row per receiver,
 * CSR) and by the sender-stationary one (w, Y, one x row per sender, out zero-filled plus one
 * out-row read-modify-write per edge, transposed CSR).  *choice = the smaller (receiver on a
 * tie).  Host only.  Any output pointer may be NULL. */
uvu_status uvu_conv_fwd_model(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, uvu_fwd_mode *choice,
                              double *bytes_receiver, double *bytes_sender);

/* Sender-stationary forward: the same out as uvu_conv_fwd, formed by one thread per (sender,
 * channel) that keeps its x row in registers, walks the sender's out-edges over the transposed
 * CSR (send_offsets, send_eids, send_recv of uvu_csr_transpose) and adds each edge's
 * contribution to out[recv] with reduction atomics after zero-filling out.  The summation order
 * varies between runs (fp32 results differ in the last bits; within the same tolerance).
 * Launches: 1 memset + 1 kernel. */
uvu_status uvu_conv_fwd_sender(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                               const void *Y, const void *w, const int32_t *send_offsets,
                               const int32_t *send_eids, const int32_t *send_recv, void *out,
                               uvu_stream_t stream);

/* Forward by mode: UVU_FWD_RECEIVER = uvu_conv_fwd (needs recv_offsets, src), UVU_FWD_SENDER =
 * uvu_conv_fwd_sender (needs the transposed CSR), UVU_FWD_AUTO = the one uvu_conv_fwd_model
 * chooses (the arrays of the other mode may be NULL). */
uvu_status uvu_conv_fwd_mode(uvu_plan_t plan, uvu_fwd_mode mode, int64_t n_nodes, int64_t n_edges,
                             const void *x, const void *Y, const void *w, const int32_t *recv_offsets,
                             const int32_t *src, const int32_t *send_offsets, const int32_t *send_eids,
                             const int32_t *send_recv, void *out, uvu_stream_t stream);

/* --------------------------- channel mixing: factorised UVW convolutions reduced to UVU ---- */

/* A UVW path whose per-edge weights factor as W_e[p,u,w] = w[e,p,u] * M[p,u,w], with the channel
 * mixing M [P][U][W] shared by all edges, reduces to the UVU convolution followed by the mixing,
 * applied once per receiver because it commutes with the sum over a receiver's edges
 * ("Receiver-streaming convolutions ...", replies: UVW cases that can be reduced to UVU; which
 * cases is not stated there, this factorisation is the reading taken):
 *     out[r,w,ooff(p)+m3] = sum_u M[p,u,w] in[r,u,ooff(p)+m3]
 * in [N][U][D_out] (a UVU output), out [N][W][D_out], W = w_out in [1, 4096].  The kernels copy
 * the operand to a component-major layout in `workspace` (at least the forward size
 * uvu_mix_workspace() reports), run one dense product per path, and copy the result back.
 * Caller-owned device memory, 16-byte aligned; out is overwritten.  Launches: 3 kernels. */
uvu_status uvu_mix_fwd(uvu_plan_t plan, int64_t n_nodes, int w_out, const void *in, const void *M,
                       void *out, void *workspace, size_t workspace_bytes, uvu_stream_t stream);

/* VJP of uvu_mix_fwd for the cotangent d_out [N][W][D_out]: d_in [N][U][D_out] and
 * dM [P][U][W] = sum_r sum_m3 in[r,u,ooff+m3] d_out[r,w,ooff+m3]; either may be NULL.  dM is a
 * product over fixed row chunks (fp32 within 16 rows, fp64 across) added in chunk
 * order: deterministic.  `workspace` holds at least the backward size of uvu_mix_workspace().
 * For N = 0, dM is set to zero.  Launches: 4 kernels for d_in, 4 for dM. */
uvu_status uvu_mix_bwd(uvu_plan_t plan, int64_t n_nodes, int w_out, const void *in, const void *M,
                       const void *d_out, void *d_in, void *dM, void *workspace, size_t workspace_bytes,
                       uvu_stream_t stream);

/* Device workspace bytes of uvu_mix_fwd and uvu_mix_bwd (either pointer may be NULL). */
uvu_status uvu_mix_workspace(uvu_plan_t plan, int64_t n_nodes, int w_out, size_t *fwd_bytes,
                             size_t *bwd_bytes);

/* The factorised UVW convolution: uvu_conv_fwd into uvu_out [N][U][D_out] (caller-owned), then
 * uvu_mix_fwd into out [N][W][D_out] with `workspace` (the forward size of uvu_mix_workspace()).
 * Its VJP composes uvu_mix_bwd (d_in is the convolution's d_out) with uvu_conv_bwd.
 * Launches: 4 kernels. */
uvu_status uvu_conv_uvw_fwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                            const void *Y, const void *w, const int32_t *recv_offsets,
                            const int32_t *src, const void *M, int w_out, void *uvu_out, void *out,
                            void *workspace, size_t workspace_bytes, uvu_stream_t stream);

/* ------------------------------------------------------- batched tensor product (no graph) ---- */

/* The channel-wise CG tensor product on its own, over a batch of B independent samples ("An
 * Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks", abstract: two dense
 * feature vectors contracted with a structured sparse tensor, before its fusion with a graph
 * convolution), with the plan's paths and coefficients:
 *     out[b,u,ooff(p)+m3] = w[.,p,u] * sum_{m1,m2} C^p[m1,m2,m3] x[b,u,xoff(p)+m1] y[b,yoff(p)+m2]
 * x [B][U][D_x], y [B][D_Y], out [B][U][D_out] in the convolution's layouts.  w is per sample,
 * [B][P][U] (w_shared = 0), or shared by the batch, [P][U] (w_shared != 0).  Every tensor is
 * caller-owned device memory, 16-byte aligned; out is overwritten (B = 0 writes nothing).
 * It runs the plan's pipelined receiver kernels with sample b as receiver b holding the one edge
 * b from sender b, so it needs a plan with U >= 32 (UVU_ERR_UNSUPPORTED otherwise).  The kernels
 * are compiled on the first call for each weight mode (host, NVRTC) and loaded once per device.
 * Launches: 1 kernel. */
uvu_status uvu_tp_fwd(uvu_plan_t plan, int64_t batch, const void *x, const void *y, const void *w,
                      int w_shared, void *out, uvu_stream_t stream);

/* VJP of uvu_tp_fwd for the cotangent d_out [B][U][D_out]: dx [B][U][D_x], dy [B][D_Y] and dw
 * ([B][P][U] per sample, or [P][U] summed over the batch when w_shared); any may be NULL = not
 * computed.  A shared dw is formed deterministically and in fp64: each block of the edge kernel
 * sums its samples in order into one fp64 row of `workspace` (at least uvu_tp_bwd_workspace()
 * bytes), then the rows are added in block order and rounded once to the plan's type.  For
 * B = 0 a shared dw is set to zero.
 * Launches: 1 kernel, plus the row sum for a shared dw. */
uvu_status uvu_tp_bwd(uvu_plan_t plan, int64_t batch, const void *x, const void *y, const void *w,
                      int w_shared, const void *d_out, void *dx, void *dy, void *dw, void *workspace,
                      size_t workspace_bytes, uvu_stream_t stream);

/* Bytes of device workspace uvu_tp_bwd needs (0 unless w_shared): min(B, 2048) * P * U * 8. */
uvu_status uvu_tp_bwd_workspace(uvu_plan_t plan, int64_t batch, int w_shared, size_t *bytes);

/* -------------------------------------------------------------- fused radial weights ---- */

/* Radial network of the fused-weight convolution ("Receiver-streaming convolutions for
 * channel-wise UVU tensor products", replies: the radial weights are materialised by a separate
 * network before the convolution; fusing that network into it is named as the next step).  The
 * page does not give the network; the one here is the radial network of MACE-style potentials.
 * For each edge e with length r[e] > 0:
 *     b_n   = sqrt(2 / r_cut) sin(n pi r / r_cut) / r * f(r / r_cut),   n = 1 .. widths[0]
 *     f(s)  = 1 - (p+1)(p+2)/2 s^p + p(p+2) s^(p+1) - p(p+1)/2 s^(p+2) for s < 1, 0 otherwise
 *     a_0 = b,  a_i = silu(a_(i-1) W_i) for i = 1 .. n_layers,  h[e] = a_(n_layers)
 * with p = p_env and silu(v) = v / (1 + exp(-v)), no biases.  The last linear layer (hidden ->
 * P x U) is not applied here: uvu_conv_fwd_radial applies it.
 * r [E] and h [E][widths[n_layers]] are device memory of the plan's type; `weights` is device
 * memory holding W_1 .. W_n_layers back to back, each row-major [widths[i-1]][widths[i]];
 * `widths` is a host array of n_layers + 1 entries.  Limits: 1 <= n_layers <= 4,
 * 1 <= widths[0] <= 64, later widths multiples of 4 in [4, 128], 1 <= p_env <= 16, r_cut > 0
 * (UVU_ERR_INVALID_ARGUMENT otherwise).  Pointers 16-byte aligned; h is overwritten.
 * Edges at or beyond r_cut get h = 0 (every layer maps 0 to 0).  Launches: 1 kernel. */
uvu_status uvu_radial_hidden(uvu_plan_t plan, int64_t n_edges, const void *r, double r_cut, int p_env,
                             int n_layers, const int *widths, const void *weights, void *h,
                             uvu_stream_t stream);

/* The convolution with fused radial weights: out = uvu_conv_fwd with
 *     w[e,p,u] = sum_k h[e,k] w_last[k,p,u]
 * formed in registers per (edge, channel) and never stored.  h [E][hidden] (uvu_radial_hidden's
 * output), w_last [hidden][P][U]; the other arguments, layouts and the CSR are those of
 * uvu_conv_fwd.  `hidden` is a multiple of 4 in [4, 256].  The kernel is generated for the
 * plan's paths and for `hidden` on the first call (host, NVRTC); a plan serves one hidden width
 * (a later call with another returns UVU_ERR_UNSUPPORTED).  Receivers without edges get zero
 * rows.  Pointers 16-byte aligned (index arrays 4-byte); out is overwritten.
 * Launches: 1 kernel. */
uvu_status uvu_conv_fwd_radial(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void *x,
                               const void *Y, const void *h, int hidden, const void *w_last,
                               const int32_t *recv_offsets, const int32_t *src, void *out,
                               uvu_stream_t stream);

/* The last linear layer of the radial network, materialised: w[e,p,u] = sum_k h[e,k] w_last[k,p,u]
 * ("Receiver-streaming convolutions ...", replies: radial weights materialised by the network
 * before the convolution).  h [E][hidden], w_last [hidden][P][U], w [E][P][U], device memory of the
 * plan's type, 16-byte aligned; w is overwritten.  fp32 plans run it on the tensor cores
 * (tcgen05, each operand split into two TF32 parts, three products per term: fp32 accuracy);
 * fp64 plans on CUDA cores.  On GB300 this at HBM speed, followed by uvu_conv_fwd, is faster than
 * the fused uvu_conv_fwd_radial, which forms every weight on CUDA cores; the fused form needs no
 * memory for w.  `hidden` is a multiple of 4 in [4, 256].  `workspace`: caller-owned device
 * memory of at least uvu_radial_weights_workspace() bytes, 16-byte aligned (w_last split into
 * its tensor-core parts, about 4 bytes per element of w_last).  Launches: 2 kernels. */
uvu_status uvu_radial_weights(uvu_plan_t plan, int64_t n_edges, const void *h, int hidden, const void *w_last,
                              void *w, void *workspace, size_t workspace_bytes, uvu_stream_t stream);

/* Bytes of device workspace uvu_radial_weights needs. */
uvu_status uvu_radial_weights_workspace(uvu_plan_t plan, int hidden, size_t *bytes);

/* Gradients of the last layer for the cotangent dw [E][P][U] of w (uvu_conv_bwd's dw):
 *     dh[e,k]         = sum_{p,u} dw[e,p,u] w_last[k,p,u]      [E][hidden]
 *     dw_last[k,p,u]  = sum_e h[e,k] dw[e,p,u]                 [hidden][P][U]
 * Either output may be NULL (not computed).  dh: tensor cores for fp32 plans (the K = P*U sum is
 * split over several accumulators added in fp32 registers), CUDA cores for fp64.  dw_last, a sum
 * over all edges, runs on CUDA cores: fp32 sums of 16 edges, Kahan-compensated, fp64 partials per
 * 1024 edges added in order, so it is deterministic (the tensor memory's fp32 accumulation lost
 * too much over such sums to keep the fp32 tolerance).  `workspace`: caller-owned device memory of
 * at least uvu_radial_weights_bwd_workspace() bytes, 16-byte aligned.  n_edges == 0 sets dw_last
 * to zero.  Launches: 2 kernels for dh, 2 for dw_last. */
uvu_status uvu_radial_weights_bwd(uvu_plan_t plan, int64_t n_edges, const void *h, int hidden, const void *w_last,
                                  const void *dw, void *dh, void *dw_last, void *workspace, size_t workspace_bytes,
                                  uvu_stream_t stream);

/* Bytes of device workspace uvu_radial_weights_bwd needs. */
uvu_status uvu_radial_weights_bwd_workspace(uvu_plan_t plan, int64_t n_edges, int hidden, size_t *bytes);

/* Reverse pass of the radial network of uvu_radial_hidden for the cotangent dh [E][widths[n]] of h:
 *     dr[e]     = d/dr_e <dh, h>            (the edge-length gradient that forces need)
 *     dweights  = d/dW_i <dh, h>, i = 1..n  (same layout as `weights`: W_1 .. W_n back to back)
 * Each tile of edges recomputes the forward pass in shared memory, then applies the chain rule
 * through the SiLU layers, the envelope and the Bessel basis.  dweights sums over all edges:
 * compensated (Kahan) fp32 sums per block in `workspace`, added over the blocks in fp64 in block
 * order (deterministic).  Arguments as uvu_radial_hidden; dr [E] and dweights are overwritten
 * (edges at or beyond r_cut get dr = 0).  `workspace`: at least
 * uvu_radial_hidden_bwd_workspace() bytes, 16-byte aligned.  UVU_ERR_UNSUPPORTED when the network's
 * activations do not fit the block's shared memory even with 16-edge tiles.  n_edges == 0 sets
 * dweights to zero.  Launches: 2 kernels. */
uvu_status uvu_radial_hidden_bwd(uvu_plan_t plan, int64_t n_edges, const void *r, double r_cut, int p_env,
                                 int n_layers, const int *widths, const void *weights, const void *dh, void *dr,
                                 void *dweights, void *workspace, size_t workspace_bytes, uvu_stream_t stream);

/* Bytes of device workspace uvu_radial_hidden_bwd needs on the current device. */
uvu_status uvu_radial_hidden_bwd_workspace(uvu_plan_t plan, int64_t n_edges, int n_layers, const int *widths,
                                           size_t *bytes);

/* Generated source and compile log of the fused radial forward for `hidden`, built on the host
 * if it is not yet (this fixes the plan's hidden width, as a first uvu_conv_fwd_radial does).
 * The strings stay valid for the plan's lifetime. */
uvu_status uvu_radial_module_source(uvu_plan_t plan, int hidden, const char **source, const char **log);

/* ------------------------------------------------------------------------ measurement ---- */

/* Arithmetic-rate probe, the denominator of the FP32 / FP64 pipe fractions that the benchmark
 * reports beside the HBM fractions (the pages give no peak for the hardware used here; the
 * fraction of a pipe's peak is this library's own measurement): blocks x 256 threads, each
 * running 8 independent FMA chains of `iters` steps (rounded up to a multiple of 4) in the
 * dtype.  out: device memory of at least blocks * 256 elements of the dtype (16-byte aligned),
 * overwritten with each thread's chain sum.  *fmas (host, may be NULL) receives the number of
 * FMAs one launch performs (2 flop each).  Launches: 1 kernel. */
uvu_status uvu_fma_rate_probe(uvu_dtype dtype, int blocks, int iters, void *out, double *fmas,
                              uvu_stream_t stream);

/* ---------------------------------------------------------------------------- errors ---- */

const char *uvu_status_string(uvu_status s);
const char *uvu_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* UVU_H_ */
