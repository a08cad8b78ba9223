/*
 * moonep.h -- C ABI of the GB300 (sm_103a) MoonEP layer path.
 *
 * R expert-parallel ranks are simulated as partitions of one GPU's memory.
 * One MoE layer runs as six stream-ordered calls:
 *
 *   moonep_plan              histogram + constructive balancing plan + per-copy
 *                            destinations (all on the device, no host sync)
 *   moonep_prefetch_weights  copy home expert weights into the prefetch slots
 *   moonep_dispatch          fused permute: every token copy to its final row
 *   moonep_grouped_gemm      Y = recv x W over the [E+B, H, H'] weight rows
 *   moonep_combine           fused unpermute, weighted by the top-K gates
 *   moonep_reduce_grad       fold the slot gradients back into the home rows
 *
 * and its backward: moonep_combine_backward, moonep_grouped_gemm_dx,
 * moonep_grouped_gemm_dw (which writes the slot gradients reduce_grad folds)
 * and moonep_dispatch_backward.
 *
 * Symbols: R ranks, E experts, L = E/R experts homed on each rank
 * (home(e) = e / L), B prefetch slots per rank, K experts per token, S tokens
 * per rank, C = S*K copies per rank, N = R*C copies in all, H the hidden size,
 * Hp = H' the expert FFN width.
 *
 * Conventions for every call
 *  - Memory: the caller allocates and frees every buffer, including the plan
 *    workspace.  The library never allocates, frees or synchronises, except
 *    moonep_read_status and moonep_plan_export, which say so.
 *  - Pointers are device pointers unless stated; each must be 16-byte aligned
 *    (MOONEP_ERR_ALIGN otherwise).  bf16 values are passed as their 16-bit
 *    patterns (uint16_t).  Arrays are dense, row-major, no padding.
 *  - stream is a cudaStream_t (NULL = legacy default stream).  All work is
 *    enqueued on it; shapes and launch configurations depend only on the dims,
 *    never on routing, so a sequence of calls can be captured in a CUDA graph.
 *  - Return value: a host-detected status (0 = MOONEP_OK), returned before
 *    anything is enqueued.  Conditions only the device can see (bad routing,
 *    a device wait that ran out) are OR-ed into a status word inside the plan
 *    workspace; every later kernel that uses that plan then returns without
 *    writing anything.  Read it with moonep_read_status.
 */
#ifndef MOONEP_H
#define MOONEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moonep_dims {
  int32_t R, E, B, K, S, H, Hp;
  int32_t mode;   /* 0 = training (requires B >= E/R), 1 = inference (B >= 0) */
  int32_t policy; /* planner choice among the plans Theorem 1 allows:
                     0 = the smallest-id underloaded rank from the smallest-id
                         overloaded rank, donor experts in descending id;
                     1 = largest first: the rank with the largest deficit from
                         the rank with the largest surplus, donor experts in
                         descending remaining copies (fewest distinct experts
                         per fill) */
  int32_t gemm_rows; /* height of the grouped GEMMs' work tiles ("Kimi K3 模型结构（8）",
                        rank 内部: the schedule's parameters are fixed from the load
                        before the GEMM runs):
                        0 = chosen on the device at every plan by an analytic
                            cost model over the plan's actual group sizes,
                        128 or 256 = fixed (other values: MOONEP_ERR_ARG) */
} moonep_dims;

enum moonep_status {
  MOONEP_OK = 0,
  MOONEP_ERR_ARG = 1,      /* null pointer, non-positive dimension, bad mode, policy or gemm_rows */
  MOONEP_ERR_ALIGN = 2,    /* a pointer is not 16-byte aligned                 */
  MOONEP_ERR_SLOTS = 3,    /* training mode with B < E/R                       */
  MOONEP_ERR_SHAPE = 4,    /* E % R != 0, K > E, E > 4096, H or Hp not a multiple
                              of 64, or N, R*B*H or E*H reaches 2^31            */
  MOONEP_ERR_CUDA = 5,     /* a CUDA runtime call or launch failed             */
  MOONEP_ERR_SCRATCH = 6,  /* moonep_plan_noalloc: the dims need more planner
                              scratch than its fixed static capacity            */
  /* device-detected bits, OR-ed into the workspace status word */
  MOONEP_ERR_ROUTING = 0x100,  /* an expert id outside [0,E) or repeated within a token */
  MOONEP_ERR_INTERNAL = 0x200, /* a planner invariant failed (cannot happen for valid routing) */
  MOONEP_ERR_TIMEOUT = 0x400   /* a bounded device-side wait gave up           */
};

/* Byte offsets of the tables inside the plan workspace (all 256-byte aligned).
 * Integer tables are int32 unless noted. */
typedef struct moonep_plan_layout {
  size_t total_bytes;
  size_t status;       /* int32[1]   sticky device status word; it opens a 256-byte
                          header (status, counters, internal GEMM work-item
                          counters) that moonep_plan zeroes                  */
  size_t counters;     /* int32[8]   n_fills, n_mtiles, n_occupied, n_reduce ... */
  size_t counts;       /* internal: int32[R][nchunk][E] per-chunk counts, then
                          bases (planner scratch; moonep_plan_noalloc leaves it
                          unwritten, so read T and load for the counts)     */
  size_t T;            /* int32[E]   copies routed to each expert                */
  size_t load;         /* int32[R]   copies routed to each home rank's experts   */
  size_t keep;         /* int32[E]   copies of e computed on its home rank       */
  size_t gidx;         /* int32[R][S][K] ordinal of each copy within its expert  */
  size_t fills;        /* int32[R-1][3] (u, o, d) in the order performed         */
  size_t slot_expert;  /* int32[R][B] expert held by slot (u,j), -1 if empty     */
  size_t n_recv;       /* int32[R]   distinct remote experts rank u computes     */
  size_t src;          /* int32[R]   the single rank u receives from, -1 if none */
  size_t cu_seqlens;   /* int32[R][E+B+1] group boundaries of each rank's buffer */
  size_t dst;          /* int32[R][S][K] destination row u*C + row of each copy  */
  size_t inverse;      /* int32[R*C] flat copy id (r*S+s)*K+k of each row        */
  size_t pieces;       /* internal: per-expert ranges of ordinals and their rows */
  size_t occupied;     /* int32[R*B] occupied slot ids u*B+j, ascending          */
  size_t reduce;       /* internal: per-expert slot lists for reduce_grad        */
  size_t mtiles;       /* internal: GEMM work tiles of 128 or 256 rows (int32[4]) */
  int32_t nchunk;      /* token chunks per rank used by the histogram            */
  int32_t max_mtiles;
  size_t route;        /* int32[R][S][K] send-once route entries: the copy's row
                          offset on its destination rank, or -offset-1 when an
                          earlier entry of the same token already goes there  */
  size_t groups;       /* internal: non-empty (rank, weight row) groups, int32[4]
                          each (first row, rows, weight row, rank)             */
} moonep_plan_layout;

/* Index of each counter in the `counters` table. */
enum moonep_counter {
  MOONEP_CNT_FILLS = 0,    /* fills performed (<= R-1)                     */
  MOONEP_CNT_MTILES = 1,   /* GEMM work tiles over all ranks and groups    */
  MOONEP_CNT_OCCUPIED = 2, /* occupied prefetch slots                      */
  MOONEP_CNT_REDUCE = 3,   /* home experts with at least one slot copy     */
  MOONEP_CNT_REMOTE_ENTRIES = 4, /* route entries whose destination is not the token's own rank */
  MOONEP_CNT_REMOTE_PAIRS = 5,   /* distinct (token, destination rank) pairs among those       */
  MOONEP_CNT_GROUPS = 6,         /* non-empty (rank, weight row) groups                         */
  MOONEP_CNT_TILE_ROWS = 7       /* work-tile height the plan chose for the GEMMs (128 or 256)  */
};

/* Size in bytes of the plan workspace for `dims` (host only, no CUDA call).
 * Returns MOONEP_ERR_* for invalid dims.  Its last MOONEP_GEMM_SCRATCH_BYTES
 * are the grouped GEMMs' scratch: per-CTA copies of tensor maps, which hold
 * the device addresses of the buffers the last GEMM call was given (so two
 * otherwise identical runs on different buffers differ there). */
#define MOONEP_GEMM_SCRATCH_BYTES (512u << 10)
int moonep_plan_workspace_bytes(const moonep_dims* dims, size_t* bytes);

/* Offsets of the workspace tables, so callers can view them (host only). */
int moonep_get_plan_layout(const moonep_dims* dims, moonep_plan_layout* out);

/* Device pointers to the plan's main tables inside a plan workspace: the
 * buffer views and cu_seqlens the pages' dispatch hands back ("Moonshot AI 开源
 * MoonEP", contract paragraph).  Host only: computed from the layout, no GPU
 * work and no synchronisation.  plan_ws is the device workspace (16-byte
 * aligned) that moonep_plan fills; the pointers stay valid as long as it does
 * and the tables hold the last plan written into it.  Returns MOONEP_ERR_ARG
 * for a NULL plan_ws or out, MOONEP_ERR_ALIGN for a misaligned plan_ws. */
typedef struct moonep_plan_view {
  const int32_t* cu_seqlens;  /* [R][E+B+1] group boundaries of each rank's buffer */
  const int32_t* dst;         /* [R][S][K] destination row u*C + row of each copy  */
  const int32_t* inverse;     /* [R*C] flat copy id (r*S+s)*K+k of each row         */
  const int32_t* slot_expert; /* [R][B] expert held by slot (u,j), -1 if empty      */
  const int32_t* status;      /* the sticky device status word                      */
} moonep_plan_view;
int moonep_plan_views(const moonep_dims* dims, const void* plan_ws, moonep_plan_view* out);

/* Plan one layer from the router's top-K output.
 *
 * Defines: the histogram, and the constructive balancing plan of Theorem 1
 * ("Kimi K3 模型结构（8）：训练并行，MoonEP 与四类等待", section 定理 1; "MoonEP :
 * l'équilibrage parfait", section Le théorème): ranks with fewer than C copies
 * on their home experts are underloaded, those with more are overloaded; the
 * underloaded rank u is filled to exactly C from one overloaded rank o (which
 * pair and which of o's experts: dims->policy), taking inside an expert the
 * copies with the highest ordinal first; o goes back to the set matching its
 * new load; at most R-1 fills and at most E/R experts per receiving rank
 * whatever the policy.  Then the buffer layout of the
 * framework contract ("Moonshot AI 开源 MoonEP", contract paragraph): rank u's
 * C rows are grouped by weight row g in [0, E+B) ascending (rows [0,E) home
 * experts, [E, E+B) slots), copies in ascending ordinal inside a group,
 * cu_seqlens[u][g] the first row of group g; and each copy's destination
 * ("在线规划、零拷贝、静态 shape": the planner fixes every copy's final position).
 * In inference mode (mode 1) received experts beyond the B slots use their
 * home row g = e on the receiving rank.
 *
 * topk_idx : int32 [R][S][K] expert ids (device, read only).
 * plan_ws  : workspace of moonep_plan_workspace_bytes (device, overwritten).
 * Routing errors set MOONEP_ERR_ROUTING in the workspace status word. */
int moonep_plan(const moonep_dims* dims, const int32_t* topk_idx, void* plan_ws,
                void* stream);

/* Fill the prefetch slots: w_slot[u][j] = w_home[slot_expert[u][j]] for every
 * occupied slot; empty slots are not written ("Moonshot AI 开源 MoonEP": rows
 * [E, E+B) are local prefetch slots filled by buffer.prefetch_weight).
 * w_home : bf16 [E][H][Hp] (read).  w_slot : bf16 [R][B][H][Hp] (written). */
int moonep_prefetch_weights(const moonep_dims* dims, void* plan_ws,
                            const uint16_t* w_home, uint16_t* w_slot, void* stream);

/* Fused permute: recv[dst[r][s][k]] = x[r][s] for every copy ("Kimi K3
 * 模型结构（8）", section 在线规划、零拷贝、静态 shape: tokens go straight to their
 * expert-grouped position in a fixed S*K buffer per rank).
 * x : bf16 [R][S][H] (read).  recv : bf16 [R][C][H] (every row written). */
int moonep_dispatch(const moonep_dims* dims, void* plan_ws, const uint16_t* x,
                    uint16_t* recv, void* stream);

/* Send-once dispatch ("Kimi K3 模型结构（8）", section 在线规划、零拷贝、静态 shape:
 * several of a token's K routes often land on the same rank, which needs the
 * token vector only once; a route entry holds its write offset on the
 * destination rank, or -offset-1 when that rank already appeared earlier in
 * the token; the send path skips the payload of negative entries and sends
 * only their 4-byte fp32 weight; the receiver copies the one row it got to the
 * other expert rows locally).  Pass 1 writes x[r][s] to the destination row of
 * every non-negative entry and every entry's gate to recv_weight at its row;
 * pass 2 copies, on each receiving rank, the row of the token's first entry
 * for that rank to the rows of its negative entries.  The final recv equals
 * moonep_dispatch's.  Uses the route table built by moonep_plan.
 * x : bf16 [R][S][H].  gates : fp32 [R][S][K].  recv : bf16 [R][C][H].
 * recv_weight : fp32 [R][C] (the weight that arrived with each row).
 * Requires K <= 128 (MOONEP_ERR_SHAPE otherwise). */
int moonep_dispatch_send_once(const moonep_dims* dims, void* plan_ws, const uint16_t* x,
                              const float* gates, uint16_t* recv, float* recv_weight,
                              void* stream);

/* Grouped GEMM over the [E+B, H, Hp] weight rows ("Moonshot AI 开源 MoonEP",
 * contract paragraph: the grouped GEMM addresses experts only by row index,
 * cu_seqlens chooses the active rows).  For each rank u and group g, rows
 * cu[u][g]..cu[u][g+1] of recv[u] are multiplied by W(u,g) = w_home[g] if
 * g < E, else w_slot[u][g-E]; fp32 accumulation, bf16 (round to nearest
 * even) output.  Tensor cores (tcgen05, TMEM accumulators, TMA-fed).
 * recv : bf16 [R][C][H].  w_home : bf16 [E][H][Hp].  w_slot : bf16
 * [R][B][H][Hp] (may be NULL when B == 0).  y : bf16 [R][C][Hp] (written).
 * Requires H % 64 == 0 and Hp % 64 == 0 (else MOONEP_ERR_SHAPE). */
int moonep_grouped_gemm(const moonep_dims* dims, void* plan_ws, const uint16_t* recv,
                        const uint16_t* w_home, const uint16_t* w_slot, uint16_t* y,
                        void* stream);

/* Fused unpermute/combine: out[r][s] = bf16( sum over k ascending of
 * gates[r][s][k] * y[dst[r][s][k]] ), fp32 accumulation ("Kimi K3 模型结构（8）",
 * section 在线规划、零拷贝、静态 shape: every (token, expert) pair carries its own
 * fp32 router weight, applied to that expert's output at combine).
 * y : bf16 [R][C][Hp].  gates : fp32 [R][S][K].  out : bf16 [R][S][Hp]. */
int moonep_combine(const moonep_dims* dims, void* plan_ws, const uint16_t* y,
                   const float* gates, uint16_t* out, void* stream);

/* reduce_grad ("Moonshot AI 开源 MoonEP", contract paragraph: slot gradients
 * live in separate reduce buffers seen as one [R, B, H, Hp] view; each home
 * expert's gradient receives the slots holding it, and consumed slots are
 * zeroed).  For every expert e with occupied slots (u,j), ascending (u,j):
 * g_home[e] += g_slot[u][j] in fp32, then g_slot[u][j] = +0.0.  Unoccupied
 * slots are not touched.
 * g_home : fp32 [E][H][Hp] (updated).  g_slot : fp32 [R][B][H][Hp] (updated). */
int moonep_reduce_grad(const moonep_dims* dims, void* plan_ws, float* g_home,
                       float* g_slot, void* stream);

/* ---- backward of the layer ------------------------------------------------
 * The routed-expert backward that produces the slot gradients reduce_grad
 * folds ("Moonshot AI 开源 MoonEP", contract paragraph: training keeps fp32
 * [E+B, H, H'] gradients whose rows [E, E+B) are separate reduce buffers;
 * "MoonEP : l'équilibrage parfait", section L'idée: in the backward pass the
 * redundant experts' gradients are staged in a local reduce buffer and
 * reduced to their home ranks afterwards).  All four use the plan of the
 * forward pass. */

/* Backward of moonep_combine: dY[dst[r][s][k]] = bf16(gates[r][s][k] *
 * d_out[r][s]) and d_gates[r][s][k] = sum over h of y[dst[r][s][k]][h] *
 * d_out[r][s][h] (fp32).  y, d_y : bf16 [R][C][Hp].  gates, d_gates : fp32
 * [R][S][K].  d_out : bf16 [R][S][Hp].  Requires K <= 128 and Hp <= 8192
 * (MOONEP_ERR_SHAPE otherwise). */
int moonep_combine_backward(const moonep_dims* dims, void* plan_ws, const uint16_t* y,
                            const float* gates, const uint16_t* d_out, uint16_t* d_y,
                            float* d_gates, void* stream);

/* Input gradient of the grouped GEMM: for each rank u and group g,
 * d_recv[rows of g] = d_y[rows of g] . W(u,g)^T (fp32 accumulation, bf16 out);
 * W(u,g) as in moonep_grouped_gemm.  d_y : bf16 [R][C][Hp].  d_recv : bf16
 * [R][C][H]. */
int moonep_grouped_gemm_dx(const moonep_dims* dims, void* plan_ws, const uint16_t* d_y,
                           const uint16_t* w_home, const uint16_t* w_slot, uint16_t* d_recv,
                           void* stream);

/* Weight gradient of the grouped GEMM: for each non-empty group (u, g),
 * G(u,g) += recv[rows of g]^T . d_y[rows of g] in fp32, where G(u,g) is
 * g_home[g] for a home group and g_slot[u][g-E] for a slot group; reduce_grad
 * then folds the slots into their home rows.  recv : bf16 [R][C][H].
 * g_home : fp32 [E][H][Hp], g_slot : fp32 [R][B][H][Hp] (both updated).
 * Training mode only (MOONEP_ERR_ARG in mode 1); H must be a multiple of 128
 * (MOONEP_ERR_SHAPE). */
int moonep_grouped_gemm_dw(const moonep_dims* dims, void* plan_ws, const uint16_t* recv,
                           const uint16_t* d_y, float* g_home, float* g_slot, void* stream);

/* Backward of moonep_dispatch: d_x[r][s] = bf16( sum over k ascending of
 * d_recv[dst[r][s][k]] ) (fp32 sums).  d_recv : bf16 [R][C][H].  d_x : bf16
 * [R][S][H]. */
int moonep_dispatch_backward(const moonep_dims* dims, void* plan_ws, const uint16_t* d_recv,
                             uint16_t* d_x, void* stream);

/* Copy the workspace status word to *host_status.  SYNCHRONISES the stream. */
int moonep_read_status(const moonep_dims* dims, const void* plan_ws,
                       int32_t* host_status, void* stream);

/* Copy the whole workspace to host memory (host_dst, total_bytes long), for
 * tests and debugging.  SYNCHRONISES the stream. */
int moonep_plan_export(const moonep_dims* dims, const void* plan_ws, void* host_dst,
                       void* stream);

/* Text for a status code (host or device bits). */
const char* moonep_status_string(int status);

/* Number of kernels this library has launched in this process. */
uint64_t moonep_launch_count(void);

/* Self-test of the device-side bounded wait used by the GEMM pipeline (no
 * counterpart on the pages; failure-detection support).  Launches one tiny
 * kernel that waits on an mbarrier nothing ever arrives on, with the GEMM's
 * wait helper and a limit of limit_us microseconds (1 .. 1,000,000); when the
 * limit expires it ORs MOONEP_ERR_TIMEOUT into *dev_status, writes the time it
 * waited to *dev_elapsed_us and returns, leaving the context usable.
 * dev_status, dev_elapsed_us : int32 device words (4-byte aligned). */
int moonep_selftest_bounded_wait(int32_t* dev_status, uint32_t limit_us, int32_t* dev_elapsed_us,
                                 void* stream);

/* moonep_plan for callers that cannot allocate device memory.
 *
 * There is no counterpart on the pages: this is an operational variant.  Some
 * callers cannot call cudaMalloc at planning time -- for example code running
 * inside a pre-sized memory pool or arena that must not grow, or a caching
 * allocator that forbids new allocations after warm-up.  This entry point computes exactly
 * what moonep_plan computes (same workspace layout, same output tables, bit
 * for bit) but keeps the planner's internal scratch -- the per-chunk expert
 * counts, the per-expert migrated ranges and their row bases, and the per-rank
 * tile offsets -- in one file-scope static device array of 4 MiB
 * (MOONEP_NOALLOC_SCRATCH_BYTES) instead of in plan_ws.  The array is part of
 * the library's device image: every GPU that loads the library holds it until
 * the process exits, and nothing is ever allocated or freed by this call (no
 * cudaMalloc, cudaFree or allocating library routine).
 *
 * Arguments are those of moonep_plan; plan_ws still receives every output
 * table (its internal scratch regions, `counts` among them, are left
 * untouched).  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and keeps it for
 * the life of the process.  A cudaDeviceReset of that device invalidates the kept address, so this
 * entry point must not be called on a device after it has been reset.
 * Every call shares the one array, which keeps the last call's contents:
 * calls whose kernels overlap on the GPU (two streams, or two host threads)
 * race on it and must be serialised by the caller.  Every scratch entry a
 * call reads is written earlier in the same call, so no clearing is needed.
 * Returns MOONEP_ERR_SCRATCH, before anything is enqueued, when the dims need
 * more than the capacity (roughly 4*(R*ceil(S/ceil(4096/K))*E + 5*E*R + E)
 * bytes plus alignment). */
#define MOONEP_NOALLOC_SCRATCH_BYTES (4u << 20)
int moonep_plan_noalloc(const moonep_dims* dims, const int32_t* topk_idx, void* plan_ws,
                        void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOONEP_H */
