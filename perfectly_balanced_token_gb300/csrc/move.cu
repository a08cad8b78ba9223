// Memory-bound kernels of the layer path: weight prefetch into slots, fused
// permute (dispatch), fused unpermute/combine and reduce_grad.
//
// All four move 16-byte vectors with streaming cache hints; each thread issues
// all of its loads before any dependent store so enough bytes are in flight to
// keep HBM busy.  Work that depends on the plan (occupied slots, experts with
// slot gradients) is read from the device-side plan; the grids are fixed by
// the dims so no host synchronisation is needed.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moonep {

// ---------------------------------------------------------------------------
// prefetch: w_slot[s] = w_home[slot_expert[s]] for every occupied slot s
// ("Moonshot AI 开源 MoonEP", contract paragraph: rows [E, E+B) are local prefetch
// slots filled before the expert GEMM)
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyVec = 4;                                   // uint4 per thread per item
constexpr int kCopyChunk = kCopyThreads * kCopyVec * 16;      // 16 KiB per work item

// Each thread loads its share of the CTA's next item before it stores the
// current one, so two items' loads are in flight per thread.  With eight
// occupied slots (0.47 GB at the pages shape) the copy lasts about 75 us, and
// launch and ramp take a visible share of it; small items on a grid of 16
// CTAs per SM keep the last round of items short (measured: 2-3 % faster than
// 32 KiB items loaded and stored in turn).
__global__ void __launch_bounds__(kCopyThreads)
k_prefetch(Dims d, PlanPtrs p, const uint4* __restrict__ w_home, uint4* __restrict__ w_slot) {
  if (plan_failed(p.status)) return;
  const size_t vec_per_w = (size_t)d.H * d.Hp * 2 / 16;
  const int nch = (int)((vec_per_w * 16 + kCopyChunk - 1) / kCopyChunk);
  const int items = p.counters[MOONEP_CNT_OCCUPIED] * nch;
  uint4 v[kCopyVec], nv[kCopyVec];
  auto load = [&](int it, uint4 (&r)[kCopyVec]) {
    const int e = p.slot_expert[p.occupied[it / nch]];
    const size_t v0 = (size_t)(it % nch) * (kCopyChunk / 16);
    const uint4* src = w_home + (size_t)e * vec_per_w;
#pragma unroll
    for (int i = 0; i < kCopyVec; ++i) {
      const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
      if (a < vec_per_w) r[i] = __ldcs(src + a);
    }
  };
  int it = blockIdx.x;
  if (it < items) load(it, v);
  for (; it < items; it += gridDim.x) {
    const int next = it + gridDim.x;
    if (next < items) load(next, nv);
    const int s = p.occupied[it / nch];
    const size_t v0 = (size_t)(it % nch) * (kCopyChunk / 16);
    uint4* dst = w_slot + (size_t)s * vec_per_w;
#pragma unroll
    for (int i = 0; i < kCopyVec; ++i) {
      const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
      if (a < vec_per_w) __stcs(dst + a, v[i]);
    }
#pragma unroll
    for (int i = 0; i < kCopyVec; ++i) v[i] = nv[i];
  }
}

// ---------------------------------------------------------------------------
// dispatch: recv[dst[r,s,k]] = x[r,s] -- one token row is read once and
// written K times ("Kimi K3 模型结构（8）", section 在线规划、零拷贝、静态 shape)
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 128;

template <int VPT>
__global__ void __launch_bounds__(kRowThreads)
k_dispatch(Dims d, PlanPtrs p, const uint4* __restrict__ x, uint4* __restrict__ recv) {
  if (plan_failed(p.status)) return;
  const int hv = d.H / 8;  // uint4 per row
  const int ntok = d.R * d.S;
  // the next token's row is loaded while the current one is stored
  int t = blockIdx.x;
  uint4 v[VPT], nv[VPT];
  if (t < ntok) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int a = threadIdx.x + i * kRowThreads;
      if (a < hv) v[i] = __ldcs(x + (size_t)t * hv + a);
    }
  }
  for (; t < ntok; t += gridDim.x) {
    const int tn = t + gridDim.x;
    if (tn < ntok) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int a = threadIdx.x + i * kRowThreads;
        if (a < hv) nv[i] = __ldcs(x + (size_t)tn * hv + a);
      }
    }
    const int32_t* dt = p.dst + (size_t)t * d.K;
    for (int k = 0; k < d.K; ++k) {
      uint4* out = recv + (size_t)__ldg(dt + k) * hv;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int a = threadIdx.x + i * kRowThreads;
        if (a < hv) __stcs(out + a, v[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) v[i] = nv[i];
  }
}

// ---------------------------------------------------------------------------
// send-once dispatch, two passes ("Kimi K3 模型结构（8）", section 在线规划、零拷贝、
// 静态 shape): the send pass writes a token's payload once per destination rank
// (entries with route >= 0) and every entry's fp32 weight; the receive pass
// replicates, on the destination rank, the row that arrived to the rows of the
// token's later entries for that rank (route < 0).
// ---------------------------------------------------------------------------
template <int VPT>
__global__ void __launch_bounds__(kRowThreads)
k_send(Dims d, PlanPtrs p, const uint4* __restrict__ x, const float* __restrict__ gates,
       uint4* __restrict__ recv, float* __restrict__ recv_w) {
  if (plan_failed(p.status)) return;
  const int hv = d.H / 8;
  const int ntok = d.R * d.S;
  for (int t = blockIdx.x; t < ntok; t += gridDim.x) {
    const int32_t* dt = p.dst + (size_t)t * d.K;
    const int32_t* rt = p.route + (size_t)t * d.K;
    if (threadIdx.x < d.K) {  // weights travel with every entry
      const int k = threadIdx.x;
      recv_w[__ldg(dt + k)] = __ldg(gates + (size_t)t * d.K + k);
    }
    const uint4* xr = x + (size_t)t * hv;
    uint4 v[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int a = threadIdx.x + i * kRowThreads;
      if (a < hv) v[i] = __ldcs(xr + a);
    }
    for (int k = 0; k < d.K; ++k) {
      const int code = __ldg(rt + k);
      if (code < 0) continue;  // payload already sent to that rank
      const int u = __ldg(dt + k) / d.C;
      uint4* out = recv + ((size_t)u * d.C + code) * hv;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int a = threadIdx.x + i * kRowThreads;
        if (a < hv) __stcs(out + a, v[i]);
      }
    }
  }
}

__global__ void __launch_bounds__(kRowThreads)
k_receive_copy(Dims d, PlanPtrs p, uint4* __restrict__ recv) {
  if (plan_failed(p.status)) return;
  const int hv = d.H / 8;
  const int ntok = d.R * d.S;
  for (int t = blockIdx.x; t < ntok; t += gridDim.x) {
    const int32_t* dt = p.dst + (size_t)t * d.K;
    const int32_t* rt = p.route + (size_t)t * d.K;
    for (int k = 1; k < d.K; ++k) {
      const int code = __ldg(rt + k);
      if (code >= 0) continue;
      const int u = __ldg(dt + k) / d.C;
      int first = -1;  // the entry of this token that carried the payload to u
      for (int j = 0; j < k && first < 0; ++j)
        if (__ldg(rt + j) >= 0 && __ldg(dt + j) / d.C == u) first = __ldg(rt + j);
      if (first < 0) continue;  // cannot happen for a plan-built route table
      const uint4* src = recv + ((size_t)u * d.C + first) * hv;
      uint4* dst = recv + ((size_t)u * d.C + (-code - 1)) * hv;
      for (int a = threadIdx.x; a < hv; a += kRowThreads) dst[a] = src[a];
    }
  }
}

// ---------------------------------------------------------------------------
// combine: out[r,s] = bf16( sum_k gates[r,s,k] * y[dst[r,s,k]] ), k ascending,
// fp32 fused multiply-add ("Kimi K3 模型结构（8）", same section: each expert
// output is scaled by its own fp32 router weight)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void fma_bf16x8(float* acc, float g, const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
  }
}

template <int KC>
__global__ void __launch_bounds__(kRowThreads)
k_combine(Dims d, PlanPtrs p, const uint4* __restrict__ y, const float* __restrict__ gates,
          uint4* __restrict__ out) {
  if (plan_failed(p.status)) return;
  const int hv = d.Hp / 8;
  const int ntok = d.R * d.S;
  for (int t = blockIdx.x; t < ntok; t += gridDim.x) {
    const int32_t* dt = p.dst + (size_t)t * d.K;
    const float* gt = gates + (size_t)t * d.K;
    for (int a = threadIdx.x; a < hv; a += kRowThreads) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int k0 = 0; k0 < d.K; k0 += KC) {
        uint4 v[KC];
        float g[KC];
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          if (k0 + k < d.K) {
            v[k] = __ldcs(y + (size_t)__ldg(dt + k0 + k) * hv + a);
            g[k] = __ldg(gt + k0 + k);
          }
        }
#pragma unroll
        for (int k = 0; k < KC; ++k)
          if (k0 + k < d.K) fma_bf16x8(acc, g[k], v[k]);
      }
      uint4 o;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      __stcs(out + (size_t)t * hv + a, o);
    }
  }
}

// ---------------------------------------------------------------------------
// backward of combine: for out[t] = sum_k g[t,k] Y[dst(t,k)],
//   dY[dst(t,k)] = bf16(g[t,k] * dout[t])   and   dg[t,k] = <Y[dst(t,k)], dout[t]>
// (fp32 products and sums).  One CTA per token; each thread keeps its slice of
// the dout row in registers; the copies are taken KC at a time, their Y loads
// all issued before the first is used; the K dot products are block reductions.
// ---------------------------------------------------------------------------
constexpr int kBwdMaxK = 128;

template <int VPT, int KC>
__global__ void __launch_bounds__(kRowThreads)
k_combine_bwd(Dims d, PlanPtrs p, const uint4* __restrict__ y, const float* __restrict__ gates,
              const uint4* __restrict__ dout, uint4* __restrict__ dy, float* __restrict__ dgates) {
  __shared__ float part[kRowThreads / 32][kBwdMaxK];
  if (plan_failed(p.status)) return;
  const int hv = d.Hp / 8;
  const int ntok = d.R * d.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = blockIdx.x; t < ntok; t += gridDim.x) {
    float o[VPT][8];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int a = threadIdx.x + i * kRowThreads;
      if (a < hv) {
        const uint4 v = __ldcs(dout + (size_t)t * hv + a);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(h[j]);
          o[i][2 * j] = f.x;
          o[i][2 * j + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) o[i][j] = 0.f;
      }
    }
    const int32_t* dt = p.dst + (size_t)t * d.K;
    const float* gt = gates + (size_t)t * d.K;
    for (int k0 = 0; k0 < d.K; k0 += KC) {
      size_t row[KC];
      float g[KC];
      uint4 v[KC][VPT];
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        row[k] = k0 + k < d.K ? (size_t)__ldg(dt + k0 + k) : 0;
        g[k] = k0 + k < d.K ? __ldg(gt + k0 + k) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < KC; ++k)
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int a = threadIdx.x + i * kRowThreads;
          if (k0 + k < d.K && a < hv) v[k][i] = __ldcs(y + row[k] * hv + a);
        }
      float dot[KC];
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        dot[k] = 0.f;
        if (k0 + k < d.K) {
#pragma unroll
          for (int i = 0; i < VPT; ++i) {
            const int a = threadIdx.x + i * kRowThreads;
            if (a < hv) {
              const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k][i]);
              uint4 w;
              __nv_bfloat162* hw = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                dot[k] = fmaf(f.x, o[i][2 * j], dot[k]);
                dot[k] = fmaf(f.y, o[i][2 * j + 1], dot[k]);
                hw[j] = __floats2bfloat162_rn(g[k] * o[i][2 * j], g[k] * o[i][2 * j + 1]);
              }
              __stcs(dy + row[k] * hv + a, w);
            }
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int k = 0; k < KC; ++k) dot[k] += __shfl_xor_sync(0xffffffffu, dot[k], off);
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < KC; ++k)
          if (k0 + k < d.K) part[warp][k0 + k] = dot[k];
      }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < d.K; k += kRowThreads) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kRowThreads / 32; ++w) sum += part[w][k];
      dgates[(size_t)t * d.K + k] = sum;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// backward of dispatch: dx[t] = bf16( sum over k ascending of dRecv[dst(t,k)] )
// (fp32 sums), the adjoint of writing x[t] to every destination row.
// ---------------------------------------------------------------------------
template <int KC>
__global__ void __launch_bounds__(kRowThreads)
k_dispatch_bwd(Dims d, PlanPtrs p, const uint4* __restrict__ drecv, uint4* __restrict__ dx) {
  if (plan_failed(p.status)) return;
  const int hv = d.H / 8;
  const int ntok = d.R * d.S;
  for (int t = blockIdx.x; t < ntok; t += gridDim.x) {
    const int32_t* dt = p.dst + (size_t)t * d.K;
    for (int a = threadIdx.x; a < hv; a += kRowThreads) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int k0 = 0; k0 < d.K; k0 += KC) {
        uint4 v[KC];
#pragma unroll
        for (int k = 0; k < KC; ++k)
          if (k0 + k < d.K) v[k] = __ldcs(drecv + (size_t)__ldg(dt + k0 + k) * hv + a);
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          if (k0 + k < d.K) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = __bfloat1622float2(h[j]);
              acc[2 * j] += f.x;
              acc[2 * j + 1] += f.y;
            }
          }
        }
      }
      uint4 o;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      __stcs(dx + (size_t)t * hv + a, o);
    }
  }
}

// ---------------------------------------------------------------------------
// reduce_grad: g_home[e] += g_slot[s] for the slots s holding e (ascending),
// then g_slot[s] = 0 ("Moonshot AI 开源 MoonEP", contract paragraph)
//
// A work item is a 256 KiB span of one expert's rows; its slot list is read
// once into shared memory, then the span is walked in 32 KiB sub-chunks with
// 8 float4 of the home row and 8 of a slot in flight per thread.
// ---------------------------------------------------------------------------
constexpr int kRedVec = 8;                                 // float4 per thread per sub-chunk
constexpr int kRedSub = kCopyThreads * kRedVec;            // float4 per sub-chunk
constexpr int kRedSpan = 8;                                // sub-chunks per work item

__global__ void __launch_bounds__(kCopyThreads)
k_reduce(Dims d, PlanPtrs p, float4* __restrict__ g_home, float4* __restrict__ g_slot) {
  extern __shared__ int32_t s_slots[];  // [R]: slots of the current expert
  if (plan_failed(p.status)) return;
  const size_t v_per = (size_t)d.H * d.Hp / 4;
  const size_t span = (size_t)kRedSub * kRedSpan;
  const int nsp = (int)((v_per + span - 1) / span);
  const int items = p.counters[MOONEP_CNT_REDUCE] * nsp;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int e = p.red_list[it / nsp];
    const int n = p.red_n[e];
    __syncthreads();  // the previous item is done with s_slots
    for (int j = threadIdx.x; j < n; j += kCopyThreads) s_slots[j] = p.red_slots[(size_t)e * d.R + j];
    __syncthreads();
    float4* home = g_home + (size_t)e * v_per;
    const size_t s0 = (size_t)(it % nsp) * span;
    const size_t s1 = s0 + span < v_per ? s0 + span : v_per;
    for (size_t v0 = s0; v0 < s1; v0 += kRedSub) {
      float4 acc[kRedVec], v[kRedVec];
      float4* sl = g_slot + (size_t)s_slots[0] * v_per;
#pragma unroll
      for (int i = 0; i < kRedVec; ++i) {
        const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
        if (a < s1) {
          acc[i] = __ldcs(home + a);
          v[i] = __ldcs(sl + a);
        }
      }
      for (int j = 0; j < n; ++j) {
        if (j > 0) {
          sl = g_slot + (size_t)s_slots[j] * v_per;
#pragma unroll
          for (int i = 0; i < kRedVec; ++i) {
            const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
            if (a < s1) v[i] = __ldcs(sl + a);
          }
        }
#pragma unroll
        for (int i = 0; i < kRedVec; ++i) {
          const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
          if (a < s1) {
            acc[i].x = acc[i].x + v[i].x;
            acc[i].y = acc[i].y + v[i].y;
            acc[i].z = acc[i].z + v[i].z;
            acc[i].w = acc[i].w + v[i].w;
            __stcs(sl + a, make_float4(0.f, 0.f, 0.f, 0.f));
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kRedVec; ++i) {
        const size_t a = v0 + threadIdx.x + (size_t)i * kCopyThreads;
        if (a < s1) __stcs(home + a, acc[i]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

cudaError_t launch_prefetch(const Dims& d, const PlanPtrs& p, const void* w_home, void* w_slot,
                            cudaStream_t st, int* launches) {
  if (d.B == 0) return cudaSuccess;
  const int grid = sm_count() * 16;
  k_prefetch<<<grid, kCopyThreads, 0, st>>>(d, p, (const uint4*)w_home, (uint4*)w_slot);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const Dims& d, const PlanPtrs& p, const void* x, void* recv,
                            cudaStream_t st, int* launches) {
  const int hv = d.H / 8;
  const int vpt = (hv + kRowThreads - 1) / kRowThreads;
  const int ntok = d.R * d.S;
  const int grid = min(ntok, sm_count() * 16);
  const uint4* xs = (const uint4*)x;
  uint4* rv = (uint4*)recv;
  if (vpt <= 1) k_dispatch<1><<<grid, kRowThreads, 0, st>>>(d, p, xs, rv);
  else if (vpt <= 2) k_dispatch<2><<<grid, kRowThreads, 0, st>>>(d, p, xs, rv);
  else if (vpt <= 4) k_dispatch<4><<<grid, kRowThreads, 0, st>>>(d, p, xs, rv);
  else if (vpt <= 8) k_dispatch<8><<<grid, kRowThreads, 0, st>>>(d, p, xs, rv);
  else if (vpt <= 16) k_dispatch<16><<<grid, kRowThreads, 0, st>>>(d, p, xs, rv);
  else return cudaErrorInvalidValue;
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_dispatch_send_once(const Dims& d, const PlanPtrs& p, const void* x,
                                      const float* gates, void* recv, float* recv_w,
                                      cudaStream_t st, int* launches) {
  const int hv = d.H / 8;
  const int vpt = (hv + kRowThreads - 1) / kRowThreads;
  const int ntok = d.R * d.S;
  const int grid = min(ntok, sm_count() * 16);
  const uint4* xs = (const uint4*)x;
  uint4* rv = (uint4*)recv;
  if (d.K > kRowThreads) return cudaErrorInvalidValue;
  if (vpt <= 1) k_send<1><<<grid, kRowThreads, 0, st>>>(d, p, xs, gates, rv, recv_w);
  else if (vpt <= 2) k_send<2><<<grid, kRowThreads, 0, st>>>(d, p, xs, gates, rv, recv_w);
  else if (vpt <= 4) k_send<4><<<grid, kRowThreads, 0, st>>>(d, p, xs, gates, rv, recv_w);
  else if (vpt <= 8) k_send<8><<<grid, kRowThreads, 0, st>>>(d, p, xs, gates, rv, recv_w);
  else if (vpt <= 16) k_send<16><<<grid, kRowThreads, 0, st>>>(d, p, xs, gates, rv, recv_w);
  else return cudaErrorInvalidValue;
  k_receive_copy<<<grid, kRowThreads, 0, st>>>(d, p, rv);
  *launches += 2;
  return cudaGetLastError();
}

cudaError_t launch_combine(const Dims& d, const PlanPtrs& p, const void* y, const float* gates,
                           void* out, cudaStream_t st, int* launches) {
  const int ntok = d.R * d.S;
  const int grid = min(ntok, sm_count() * 16);
  if (d.K >= 8)
    k_combine<8><<<grid, kRowThreads, 0, st>>>(d, p, (const uint4*)y, gates, (uint4*)out);
  else
    k_combine<4><<<grid, kRowThreads, 0, st>>>(d, p, (const uint4*)y, gates, (uint4*)out);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_combine_backward(const Dims& d, const PlanPtrs& p, const void* y,
                                    const float* gates, const void* dout, void* dy, float* dgates,
                                    cudaStream_t st, int* launches) {
  const int hv = d.Hp / 8;
  const int vpt = (hv + kRowThreads - 1) / kRowThreads;
  const int ntok = d.R * d.S;
  const int grid = min(ntok, sm_count() * 16);
  const uint4 *ys = (const uint4*)y, *os = (const uint4*)dout;
  uint4* dys = (uint4*)dy;
  if (d.K > kBwdMaxK) return cudaErrorInvalidValue;
  // KC x VPT row vectors in flight per thread: 8 for every row width
  if (vpt <= 1) k_combine_bwd<1, 8><<<grid, kRowThreads, 0, st>>>(d, p, ys, gates, os, dys, dgates);
  else if (vpt <= 2) k_combine_bwd<2, 4><<<grid, kRowThreads, 0, st>>>(d, p, ys, gates, os, dys, dgates);
  else if (vpt <= 4) k_combine_bwd<4, 2><<<grid, kRowThreads, 0, st>>>(d, p, ys, gates, os, dys, dgates);
  else if (vpt <= 8) k_combine_bwd<8, 1><<<grid, kRowThreads, 0, st>>>(d, p, ys, gates, os, dys, dgates);
  else return cudaErrorInvalidValue;
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_dispatch_backward(const Dims& d, const PlanPtrs& p, const void* drecv, void* dx,
                                     cudaStream_t st, int* launches) {
  const int ntok = d.R * d.S;
  const int grid = min(ntok, sm_count() * 16);
  if (d.K >= 8)
    k_dispatch_bwd<8><<<grid, kRowThreads, 0, st>>>(d, p, (const uint4*)drecv, (uint4*)dx);
  else
    k_dispatch_bwd<4><<<grid, kRowThreads, 0, st>>>(d, p, (const uint4*)drecv, (uint4*)dx);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_reduce(const Dims& d, const PlanPtrs& p, float* g_home, float* g_slot,
                          cudaStream_t st, int* launches) {
  if (d.B == 0) return cudaSuccess;
  const int grid = sm_count() * 8;
  k_reduce<<<grid, kCopyThreads, sizeof(int32_t) * d.R, st>>>(d, p, (float4*)g_home, (float4*)g_slot);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace moonep
