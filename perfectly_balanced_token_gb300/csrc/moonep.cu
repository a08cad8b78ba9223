// Host side of the C ABI declared in include/moonep.h: argument checks, the
// plan-workspace layout and the launches.  Nothing here allocates device
// memory; only moonep_read_status and moonep_plan_export synchronise.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moonep {
cudaError_t launch_plan(const Dims&, const int32_t*, const PlanPtrs&, cudaStream_t, int*);
cudaError_t launch_prefetch(const Dims&, const PlanPtrs&, const void*, void*, cudaStream_t, int*);
cudaError_t launch_dispatch(const Dims&, const PlanPtrs&, const void*, void*, cudaStream_t, int*);
cudaError_t launch_dispatch_send_once(const Dims&, const PlanPtrs&, const void*, const float*, void*,
                                      float*, cudaStream_t, int*);
cudaError_t launch_grouped_gemm(const Dims&, const PlanPtrs&, const void*, const void*, const void*,
                                void*, cudaStream_t, int*);
cudaError_t launch_combine(const Dims&, const PlanPtrs&, const void*, const float*, void*,
                           cudaStream_t, int*);
cudaError_t launch_reduce(const Dims&, const PlanPtrs&, float*, float*, cudaStream_t, int*);
cudaError_t launch_grouped_gemm_dx(const Dims&, const PlanPtrs&, const void*, const void*, const void*,
                                   void*, cudaStream_t, int*);
cudaError_t launch_grouped_gemm_dw(const Dims&, const PlanPtrs&, const void*, const void*, float*,
                                   float*, cudaStream_t, int*);
cudaError_t launch_combine_backward(const Dims&, const PlanPtrs&, const void*, const float*,
                                    const void*, void*, float*, cudaStream_t, int*);
cudaError_t launch_dispatch_backward(const Dims&, const PlanPtrs&, const void*, void*, cudaStream_t,
                                     int*);
cudaError_t launch_wait_selftest(int32_t*, uint32_t, int32_t*, cudaStream_t, int*);

static std::atomic<uint64_t> g_launches{0};

static int check_dims(const moonep_dims* in, Dims* d) {
  if (in == nullptr) return MOONEP_ERR_ARG;
  const moonep_dims& x = *in;
  if (x.R <= 0 || x.E <= 0 || x.K <= 0 || x.S <= 0 || x.H <= 0 || x.Hp <= 0 || x.B < 0)
    return MOONEP_ERR_ARG;
  if (x.mode != 0 && x.mode != 1) return MOONEP_ERR_ARG;
  if (x.policy != 0 && x.policy != 1) return MOONEP_ERR_ARG;
  if (x.gemm_rows != 0 && x.gemm_rows != kMmaM && x.gemm_rows != 2 * kMmaM) return MOONEP_ERR_ARG;
  if (x.E % x.R != 0 || x.K > x.E || x.E > kMaxExperts || x.B > x.E) return MOONEP_ERR_SHAPE;
  if (x.H % 64 != 0 || x.Hp % 64 != 0) return MOONEP_ERR_SHAPE;
  const int64_t N = (int64_t)x.R * x.S * x.K;
  if (N >= (int64_t(1) << 31)) return MOONEP_ERR_SHAPE;
  if ((int64_t)x.R * x.B * x.H >= (int64_t(1) << 31)) return MOONEP_ERR_SHAPE;
  if ((int64_t)x.E * x.H >= (int64_t(1) << 31)) return MOONEP_ERR_SHAPE;
  const int L = x.E / x.R;
  if (x.mode == 0 && x.B < L) return MOONEP_ERR_SLOTS;
  d->R = x.R; d->E = x.E; d->B = x.B; d->K = x.K; d->S = x.S; d->H = x.H; d->Hp = x.Hp;
  d->mode = x.mode;
  d->policy = x.policy;
  d->L = L;
  d->C = x.S * x.K;
  d->N = (int)N;
  d->chunk_tokens = std::max(1, kChunkCopies / x.K);
  d->nchunk = (x.S + d->chunk_tokens - 1) / d->chunk_tokens;
  const int64_t groups = std::min<int64_t>((int64_t)x.E + x.B, d->C);
  d->tile_m = x.gemm_rows;  // 0: the planner chooses per plan
  // room for the longer (128-row) tile list whatever is chosen
  const int64_t mt = (N + kMmaM - 1) / kMmaM + (int64_t)x.R * groups;
  if (mt >= (int64_t(1) << 31)) return MOONEP_ERR_SHAPE;
  d->max_mtiles = (int)mt;
  d->max_groups = (int)std::min<int64_t>((int64_t)x.R * groups, int64_t(1) << 30);
  return MOONEP_OK;
}

static Layout make_layout(const Dims& d) {
  Layout L{};
  moonep_plan_layout& p = L.pub;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + std::max<size_t>(bytes, 4));
    return at;
  };
  p.status = 0;     // status word and counters share the first 256 bytes
  p.counters = 64;
  off = 256;
  const size_t R = d.R, E = d.E, B = d.B, N = d.N, EB = d.E + d.B;
  p.counts = take(4 * R * d.nchunk * E);
  p.T = take(4 * E);
  p.load = take(4 * R);
  p.keep = take(4 * E);
  p.gidx = take(4 * N);
  p.fills = take(4 * 3 * std::max<size_t>(R - 1, 1));
  p.slot_expert = take(4 * R * B);
  p.n_recv = take(4 * R);
  p.src = take(4 * R);
  p.cu_seqlens = take(4 * R * (EB + 1));
  p.dst = take(4 * N);
  p.inverse = take(4 * N);
  p.route = take(4 * N);
  p.pieces = L.pieces = take(sizeof(Piece) * E * R);
  L.piece_n = take(4 * E);
  L.piece_base = take(4 * E * R);
  L.home_base = take(4 * E);
  p.occupied = take(4 * R * B);
  p.reduce = L.red_slots = take(4 * E * R);
  L.red_n = take(4 * E);
  L.red_list = take(4 * E);
  L.rank_tiles = take(4 * (R + 1));
  p.mtiles = take(sizeof(MTile) * (size_t)d.max_mtiles);
  L.rank_groups = take(4 * (R + 1));
  p.groups = take(sizeof(MTile) * (size_t)d.max_groups);
  L.tmaps = take(MOONEP_GEMM_SCRATCH_BYTES);  // last: the layout documents it as the tail
  p.total_bytes = off;
  p.nchunk = d.nchunk;
  p.max_mtiles = d.max_mtiles;
  return L;
}

static PlanPtrs resolve(const Layout& L, void* ws) {
  char* b = static_cast<char*>(ws);
  const moonep_plan_layout& p = L.pub;
  PlanPtrs q;
  q.status = (int32_t*)(b + p.status);
  q.sched = (int32_t*)(b + p.status + 128);  // inside the 256-byte header the plan zeroes
  q.counters = (int32_t*)(b + p.counters);
  q.counts = (int32_t*)(b + p.counts);
  q.T = (int32_t*)(b + p.T);
  q.load = (int32_t*)(b + p.load);
  q.keep = (int32_t*)(b + p.keep);
  q.gidx = (int32_t*)(b + p.gidx);
  q.fills = (int32_t*)(b + p.fills);
  q.slot_expert = (int32_t*)(b + p.slot_expert);
  q.n_recv = (int32_t*)(b + p.n_recv);
  q.src = (int32_t*)(b + p.src);
  q.cu = (int32_t*)(b + p.cu_seqlens);
  q.dst = (int32_t*)(b + p.dst);
  q.inverse = (int32_t*)(b + p.inverse);
  q.route = (int32_t*)(b + p.route);
  q.pieces = (Piece*)(b + L.pieces);
  q.piece_n = (int32_t*)(b + L.piece_n);
  q.piece_base = (int32_t*)(b + L.piece_base);
  q.home_base = (int32_t*)(b + L.home_base);
  q.occupied = (int32_t*)(b + p.occupied);
  q.red_slots = (int32_t*)(b + L.red_slots);
  q.red_n = (int32_t*)(b + L.red_n);
  q.red_list = (int32_t*)(b + L.red_list);
  q.rank_tiles = (int32_t*)(b + L.rank_tiles);
  q.mtiles = (MTile*)(b + p.mtiles);
  q.rank_groups = (int32_t*)(b + L.rank_groups);
  q.groups = (MTile*)(b + p.groups);
  q.tmaps = (uint8_t*)(b + L.tmaps);
  return q;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int finish(cudaError_t e, int launches) {
  g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
  return e == cudaSuccess ? MOONEP_OK : MOONEP_ERR_CUDA;
}

// Common prologue: dims, workspace pointer, alignment of the listed pointers.
#define MOONEP_PROLOGUE(dims, ws)                  \
  Dims d;                                          \
  {                                                \
    const int rc_ = check_dims(dims, &d);          \
    if (rc_ != MOONEP_OK) return rc_;              \
  }                                                \
  if ((ws) == nullptr) return MOONEP_ERR_ARG;      \
  if (!aligned16(ws)) return MOONEP_ERR_ALIGN;     \
  const Layout lay = make_layout(d);               \
  const PlanPtrs P = resolve(lay, const_cast<void*>(static_cast<const void*>(ws)))

#define MOONEP_NEED(ptr)                            \
  do {                                              \
    if ((ptr) == nullptr) return MOONEP_ERR_ARG;    \
    if (!aligned16(ptr)) return MOONEP_ERR_ALIGN;   \
  } while (0)

}  // namespace moonep

using namespace moonep;

extern "C" {

int moonep_plan_workspace_bytes(const moonep_dims* dims, size_t* bytes) {
  Dims d;
  const int rc = check_dims(dims, &d);
  if (rc != MOONEP_OK) return rc;
  if (bytes == nullptr) return MOONEP_ERR_ARG;
  *bytes = make_layout(d).pub.total_bytes;
  return MOONEP_OK;
}

int moonep_get_plan_layout(const moonep_dims* dims, moonep_plan_layout* out) {
  Dims d;
  const int rc = check_dims(dims, &d);
  if (rc != MOONEP_OK) return rc;
  if (out == nullptr) return MOONEP_ERR_ARG;
  *out = make_layout(d).pub;
  return MOONEP_OK;
}

int moonep_plan_views(const moonep_dims* dims, const void* plan_ws, moonep_plan_view* out) {
  Dims d;
  const int rc = check_dims(dims, &d);
  if (rc != MOONEP_OK) return rc;
  if (plan_ws == nullptr || out == nullptr) return MOONEP_ERR_ARG;
  if (!aligned16(plan_ws)) return MOONEP_ERR_ALIGN;
  const moonep_plan_layout L = make_layout(d).pub;
  const uint8_t* b = static_cast<const uint8_t*>(plan_ws);
  out->cu_seqlens = reinterpret_cast<const int32_t*>(b + L.cu_seqlens);
  out->dst = reinterpret_cast<const int32_t*>(b + L.dst);
  out->inverse = reinterpret_cast<const int32_t*>(b + L.inverse);
  out->slot_expert = reinterpret_cast<const int32_t*>(b + L.slot_expert);
  out->status = reinterpret_cast<const int32_t*>(b + L.status);
  return MOONEP_OK;
}

int moonep_plan(const moonep_dims* dims, const int32_t* topk_idx, void* plan_ws, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(topk_idx);
  int n = 0;
  const cudaError_t e = launch_plan(d, topk_idx, P, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_prefetch_weights(const moonep_dims* dims, void* plan_ws, const uint16_t* w_home,
                            uint16_t* w_slot, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(w_home);
  if (d.B > 0) MOONEP_NEED(w_slot);
  int n = 0;
  const cudaError_t e = launch_prefetch(d, P, w_home, w_slot, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_dispatch(const moonep_dims* dims, void* plan_ws, const uint16_t* x, uint16_t* recv,
                    void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(x);
  MOONEP_NEED(recv);
  int n = 0;
  const cudaError_t e = launch_dispatch(d, P, x, recv, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_dispatch_send_once(const moonep_dims* dims, void* plan_ws, const uint16_t* x,
                              const float* gates, uint16_t* recv, float* recv_weight,
                              void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(x);
  MOONEP_NEED(gates);
  MOONEP_NEED(recv);
  MOONEP_NEED(recv_weight);
  if (d.K > 128) return MOONEP_ERR_SHAPE;  // one thread per route entry in the send pass
  int n = 0;
  const cudaError_t e = launch_dispatch_send_once(d, P, x, gates, recv, recv_weight,
                                                  (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_grouped_gemm(const moonep_dims* dims, void* plan_ws, const uint16_t* recv,
                        const uint16_t* w_home, const uint16_t* w_slot, uint16_t* y,
                        void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(recv);
  MOONEP_NEED(w_home);
  MOONEP_NEED(y);
  if (d.B > 0) MOONEP_NEED(w_slot);
  int n = 0;
  const cudaError_t e = launch_grouped_gemm(d, P, recv, w_home, w_slot, y, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_combine(const moonep_dims* dims, void* plan_ws, const uint16_t* y, const float* gates,
                   uint16_t* out, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(y);
  MOONEP_NEED(gates);
  MOONEP_NEED(out);
  int n = 0;
  const cudaError_t e = launch_combine(d, P, y, gates, out, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_reduce_grad(const moonep_dims* dims, void* plan_ws, float* g_home, float* g_slot,
                       void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(g_home);
  if (d.B > 0) MOONEP_NEED(g_slot);
  int n = 0;
  const cudaError_t e = launch_reduce(d, P, g_home, g_slot, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_combine_backward(const moonep_dims* dims, void* plan_ws, const uint16_t* y,
                            const float* gates, const uint16_t* d_out, uint16_t* d_y,
                            float* d_gates, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(y);
  MOONEP_NEED(gates);
  MOONEP_NEED(d_out);
  MOONEP_NEED(d_y);
  MOONEP_NEED(d_gates);
  if (d.K > 128 || d.Hp > 8192) return MOONEP_ERR_SHAPE;
  int n = 0;
  const cudaError_t e = launch_combine_backward(d, P, y, gates, d_out, d_y, d_gates,
                                                (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_grouped_gemm_dx(const moonep_dims* dims, void* plan_ws, const uint16_t* d_y,
                           const uint16_t* w_home, const uint16_t* w_slot, uint16_t* d_recv,
                           void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(d_y);
  MOONEP_NEED(w_home);
  MOONEP_NEED(d_recv);
  if (d.B > 0) MOONEP_NEED(w_slot);
  int n = 0;
  const cudaError_t e = launch_grouped_gemm_dx(d, P, d_y, w_home, w_slot, d_recv,
                                               (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_grouped_gemm_dw(const moonep_dims* dims, void* plan_ws, const uint16_t* recv,
                           const uint16_t* d_y, float* g_home, float* g_slot, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(recv);
  MOONEP_NEED(d_y);
  MOONEP_NEED(g_home);
  if (d.B > 0) MOONEP_NEED(g_slot);
  if (d.mode != 0) return MOONEP_ERR_ARG;       // gradients exist in training only
  if (d.H % 128 != 0) return MOONEP_ERR_SHAPE;  // 128-row tiles of H
  int n = 0;
  const cudaError_t e = launch_grouped_gemm_dw(d, P, recv, d_y, g_home, g_slot,
                                               (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_dispatch_backward(const moonep_dims* dims, void* plan_ws, const uint16_t* d_recv,
                             uint16_t* d_x, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(d_recv);
  MOONEP_NEED(d_x);
  int n = 0;
  const cudaError_t e = launch_dispatch_backward(d, P, d_recv, d_x, (cudaStream_t)stream, &n);
  return finish(e, n);
}

int moonep_read_status(const moonep_dims* dims, const void* plan_ws, int32_t* host_status,
                       void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  if (host_status == nullptr) return MOONEP_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(host_status, P.status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return MOONEP_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? MOONEP_OK : MOONEP_ERR_CUDA;
}

int moonep_plan_export(const moonep_dims* dims, const void* plan_ws, void* host_dst, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  (void)P;
  if (host_dst == nullptr) return MOONEP_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(host_dst, plan_ws, lay.pub.total_bytes, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return MOONEP_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? MOONEP_OK : MOONEP_ERR_CUDA;
}

const char* moonep_status_string(int s) {
  switch (s) {
    case MOONEP_OK: return "ok";
    case MOONEP_ERR_ARG: return "invalid argument (null pointer, non-positive dimension, bad mode, policy or gemm_rows)";
    case MOONEP_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOONEP_ERR_SLOTS: return "training mode needs B >= E/R prefetch slots";
    case MOONEP_ERR_SHAPE: return "unsupported shape (E%R, K>E, E>4096, B>E, H or Hp not a multiple of 64, or a size >= 2^31)";
    case MOONEP_ERR_CUDA: return "CUDA runtime error or launch failure";
    case MOONEP_ERR_SCRATCH: return "dims need more planner scratch than the fixed no-allocation capacity (4 MiB)";
    default: break;
  }
  if (s & MOONEP_ERR_ROUTING) return "device: expert id out of range or repeated within a token";
  if (s & MOONEP_ERR_INTERNAL) return "device: planner invariant failed";
  if (s & MOONEP_ERR_TIMEOUT) return "device: a bounded wait in the GEMM pipeline expired";
  return "unknown status";
}

uint64_t moonep_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moonep_selftest_bounded_wait(int32_t* dev_status, uint32_t limit_us, int32_t* dev_elapsed_us,
                                 void* stream) {
  if (dev_status == nullptr || dev_elapsed_us == nullptr) return MOONEP_ERR_ARG;
  if (limit_us == 0 || limit_us > 1000000u) return MOONEP_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) || (reinterpret_cast<uintptr_t>(dev_elapsed_us) & 3u))
    return MOONEP_ERR_ALIGN;
  int n = 0;
  const cudaError_t e = launch_wait_selftest(dev_status, limit_us, dev_elapsed_us,
                                             (cudaStream_t)stream, &n);
  return finish(e, n);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moonep_plan_noalloc: the planner with its internal scratch in a static
// device array, for callers that cannot allocate device memory.
// ---------------------------------------------------------------------------
namespace moonep {

constexpr size_t kNoAllocBytes = MOONEP_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

// Lives in the library's device image on every GPU that loads it; host code
// must not use this name as an address (it is a host-side stand-in).
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocBytes / sizeof(int32_t)];

static std::mutex g_noalloc_mutex;
static void* g_noalloc_base[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current.
static int noalloc_base(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return MOONEP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_base[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MOONEP_ERR_CUDA;
    g_noalloc_base[dev] = p;
  }
  *out = g_noalloc_base[dev];
  return MOONEP_OK;
}

// Offsets of the planner's internal tables inside the static array.
struct NoAllocLayout {
  size_t counts, pieces, piece_n, piece_base, home_base, rank_tiles, rank_groups, total;
};

static NoAllocLayout noalloc_layout(const Dims& d) {
  NoAllocLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + std::max<size_t>(bytes, 4));
    return at;
  };
  const size_t R = d.R, E = d.E;
  L.counts = take(4 * R * d.nchunk * E);
  L.pieces = take(sizeof(Piece) * E * R);
  L.piece_n = take(4 * E);
  L.piece_base = take(4 * E * R);
  L.home_base = take(4 * E);
  L.rank_tiles = take(4 * (R + 1));
  L.rank_groups = take(4 * (R + 1));
  L.total = off;
  return L;
}

}  // namespace moonep

extern "C" int moonep_plan_noalloc(const moonep_dims* dims, const int32_t* topk_idx,
                                   void* plan_ws, void* stream) {
  MOONEP_PROLOGUE(dims, plan_ws);
  MOONEP_NEED(topk_idx);
  const NoAllocLayout S = noalloc_layout(d);
  if (S.total > kNoAllocBytes) return MOONEP_ERR_SCRATCH;
  void* base = nullptr;
  const int rc = noalloc_base(&base);
  if (rc != MOONEP_OK) return rc;
  char* b = static_cast<char*>(base);
  PlanPtrs Q = P;
  Q.counts = (int32_t*)(b + S.counts);
  Q.pieces = (Piece*)(b + S.pieces);
  Q.piece_n = (int32_t*)(b + S.piece_n);
  Q.piece_base = (int32_t*)(b + S.piece_base);
  Q.home_base = (int32_t*)(b + S.home_base);
  Q.rank_tiles = (int32_t*)(b + S.rank_tiles);
  Q.rank_groups = (int32_t*)(b + S.rank_groups);
  int n = 0;
  const cudaError_t e = launch_plan(d, topk_idx, Q, (cudaStream_t)stream, &n);
  return finish(e, n);
}
