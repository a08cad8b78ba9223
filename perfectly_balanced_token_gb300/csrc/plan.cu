// Planner kernels: histogram + stable ordinals, the constructive balancing
// plan, per-rank buffer tables and per-copy destinations.
//
// The construction follows Theorem 1 of "Kimi K3 模型结构（8）：训练并行，MoonEP
// 与四类等待" (section 定理 1) and "MoonEP : l'équilibrage parfait" (section Le
// théorème): fill one underloaded rank u to exactly C = S*K from one
// overloaded rank o, put o back in the matching set, repeat; each rank is
// filled at most once, so its remote copies come from one rank and touch at
// most E/R experts.  The fixed tie-break: smallest-id u and o; o's experts in
// descending id; inside an expert the highest global ordinals first.
//
// Everything stays on the device: the histogram, plan and tables are produced
// by six launches whose shapes depend only on the dims ("Kimi K3 模型结构（8）",
// section 在线规划、零拷贝、静态 shape: static shapes remove the per-layer host
// synchronisation).
#include "common.cuh"
#include "gemm_cost.cuh"

namespace moonep {

// ---------------------------------------------------------------------------
// 1. per-chunk histogram and chunk-local stable ordinals
//    grid (nchunk, R), kHistWarps warps, smem [kHistWarps][E] counters
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kHistWarps * 32)
k_hist(Dims d, const int32_t* __restrict__ idx, PlanPtrs p) {
  extern __shared__ int32_t sh[];
  const int r = blockIdx.y, chunk = blockIdx.x;
  const int t0 = chunk * d.chunk_tokens;
  const int t1 = min(d.S, t0 + d.chunk_tokens);
  const int ncopy = (t1 - t0) * d.K;
  const size_t first = ((size_t)r * d.S + t0) * d.K;
  const int32_t* ids = idx + first;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < kHistWarps * d.E; i += blockDim.x) sh[i] = 0;

  // validate: ids in range and distinct within each token
  int bad = 0;
  for (int t = threadIdx.x; t < t1 - t0; t += blockDim.x) {
    const int32_t* tok = ids + (size_t)t * d.K;
    for (int a = 0; a < d.K; ++a) {
      const int ea = tok[a];
      bad |= (ea < 0) | (ea >= d.E);
      for (int b = a + 1; b < d.K; ++b) bad |= (tok[b] == ea);
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) set_error(p.status, MOONEP_ERR_ROUTING);
    return;
  }

  // each warp owns a contiguous, 32-aligned sub-range of the chunk's copies
  const int per = ((ncopy + kHistWarps * 32 - 1) / (kHistWarps * 32)) * 32;
  const int w_lo = min(ncopy, warp * per), w_hi = min(ncopy, w_lo + per);
  int32_t* mine = sh + warp * d.E;
  for (int i = w_lo + lane; i < w_hi; i += 32) atomicAdd(&mine[ids[i]], 1);
  __syncthreads();

  // exclusive scan across warps per expert -> chunk totals
  int32_t* cnt = p.counts + ((size_t)r * d.nchunk + chunk) * d.E;
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kHistWarps; ++w) {
      const int v = sh[w * d.E + e];
      sh[w * d.E + e] = run;
      run += v;
    }
    cnt[e] = run;
  }
  __syncthreads();

  // stable ordinals: 32 copies at a time in order, equal ids ranked by lane
  int32_t* out = p.gidx + first;
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = w_lo; i0 < w_hi; i0 += 32) {
    const int i = i0 + lane;
    const bool valid = i < w_hi;
    const int e = valid ? ids[i] : d.E + lane;  // unique filler never matches
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int before = __popc(peers & lt);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (valid) base = mine[e];
    __syncwarp();
    if (valid && lane == leader) mine[e] = base + __popc(peers);
    __syncwarp();
    if (valid) out[i] = base + before;
  }
}

// ---------------------------------------------------------------------------
// 1b. chunk bases: for every expert, the exclusive prefix of its per-chunk
//     counts in ascending (rank, chunk) order -- ascending (rank, token), the
//     order of the global ordinals -- and its total T_e.  One CTA per 32
//     experts: lane = expert, so every load is one coalesced row of 32 counts;
//     warp w takes a contiguous run of the (rank, chunk) rows and the 32 runs
//     are chained by a scan in shared memory.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
k_scan(Dims d, PlanPtrs p) {
  __shared__ int32_t part[32][33];
  if (plan_failed(p.status)) return;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int rc = d.R * d.nchunk;
  const int per = (rc + 31) / 32;
  const int i0 = min(rc, w * per), i1 = min(rc, i0 + per);
  int32_t* c = p.counts + e;
  constexpr int kBatch = 8;  // loads in flight before the dependent sum / stores
  int sum = 0;
  if (e < d.E) {
    for (int b = i0; b < i1; b += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = (b + j < i1) ? c[(size_t)(b + j) * d.E] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) sum += v[j];
    }
  }
  part[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int k = 0; k < 32; ++k) {
      const int v = part[k][lane];
      part[k][lane] = run;
      run += v;
    }
    if (e < d.E) p.T[e] = run;
  }
  __syncthreads();
  if (e < d.E) {
    int run = part[w][lane];
    for (int b = i0; b < i1; b += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) v[j] = (b + j < i1) ? c[(size_t)(b + j) * d.E] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (b + j < i1) c[(size_t)(b + j) * d.E] = run;
        run += v[j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 2. single-CTA planner: loads, the fills, slots and row counts
// ---------------------------------------------------------------------------
enum : int32_t { kBalanced = 0, kUnder = 1, kOver = 2 };

// The plain policy's fills run in parallel when the extra shared arrays fit.
__host__ __device__ inline bool kParallelFills(const Dims& d) { return d.policy == 0 && d.R <= 1024; }
__host__ __device__ inline size_t plan_smem_bytes(const Dims& d) {
  return sizeof(int32_t) * (kParallelFills(d) ? (5 * (size_t)d.E + 14 * (size_t)d.R)
                                              : (3 * (size_t)d.E + 6 * (size_t)d.R));
}

__global__ void __launch_bounds__(1024)
k_plan(Dims d, PlanPtrs p) {
  extern __shared__ int32_t sh[];
  int32_t* sT = sh;                 // [E]
  int32_t* sMig = sT + d.E;         // [E]
  int32_t* sLoad = sMig + d.E;      // [R]
  int32_t* sState = sLoad + d.R;    // [R]
  int32_t* sT128 = sState + d.R;    // [R] 128-row work tiles per rank
  int32_t* sT256F = sT128 + d.R;    // [R] 256-row work tiles with more than 128 rows
  int32_t* sT256H = sT256F + d.R;   // [R] 256-row work tiles with at most 128 rows
  int32_t* sGroups = sT256H + d.R;  // [R] non-empty weight-row groups per rank
  int32_t* sPieceN = sGroups + d.R; // [E] pieces per expert so far
  // parallel fills of the plain policy (present when kParallelFills(d))
  int32_t* sOff = sPieceN + d.E;    // [E] copies of the higher-id experts of the same rank
  int32_t* sNz = sOff + d.E;        // [E] non-empty higher-id experts of the same rank
  int32_t* sGiven = sNz + d.E;      // [R] copies a rank has given so far
  int32_t* sFU = sGiven + d.R;      // [R] fill f: receiving rank
  int32_t* sFO = sFU + d.R;         // [R] fill f: giving rank
  int32_t* sFD = sFO + d.R;         // [R] fill f: copies
  int32_t* sFB = sFD + d.R;         // [R] fill f: copies its giver gave before it
  int32_t* sFZ = sFB + d.R;         // [R] fill f: giver's non-empty experts used up before it
  int32_t* sFS = sFZ + d.R;         // [R] fill f: copies placed (check)
  int32_t* sNr = sFS + d.R;         // [R] distinct experts a rank received
  if (plan_failed(p.status)) return;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int EB = d.E + d.B;

  // T from the chunk scan
  for (int e = tid; e < d.E; e += nt) {
    sT[e] = p.T[e];
    sMig[e] = 0;
    sPieceN[e] = 0;
    p.red_n[e] = 0;
  }
  for (int s = tid; s < d.R * d.B; s += nt) p.slot_expert[s] = -1;
  for (int i = tid; i < d.R * (EB + 1); i += nt) p.cu[i] = 0;
  for (int h = tid; h < d.R; h += nt) {
    p.n_recv[h] = 0;
    p.src[h] = -1;
    sT128[h] = 0;
    sT256F[h] = 0;
    sT256H[h] = 0;
    sGroups[h] = 0;
  }
  for (int i = tid; i < 3 * max(d.R - 1, 1); i += nt) p.fills[i] = -1;
  __syncthreads();
  for (int h = tid; h < d.R; h += nt) {
    int s = 0;
    for (int e = h * d.L; e < (h + 1) * d.L; ++e) s += sT[e];
    sLoad[h] = s;
    p.load[h] = s;
    sState[h] = s < d.C ? kUnder : (s > d.C ? kOver : kBalanced);
  }
  __syncthreads();

  // a non-empty group of `rows` rows on rank u: its work tiles at both heights
  auto count_group = [&](int u, int rows) {
    atomicAdd(&sT128[u], (rows + kMmaM - 1) / kMmaM);
    const int rem = rows % (2 * kMmaM);
    atomicAdd(&sT256F[u], rows / (2 * kMmaM) + (rem > kMmaM ? 1 : 0));
    if (rem > 0 && rem <= kMmaM) atomicAdd(&sT256H[u], 1);
    atomicAdd(&sGroups[u], 1);
  };

  const bool parallel_fills = kParallelFills(d);
  if (parallel_fills) {
    // Plain policy.  The fill sequence itself -- which rank fills which and
    // by how much -- depends only on the loads (warp 0, ballots); where the
    // copies come from follows without a walk: each giver's copies are taken
    // as one sequence (its experts in descending id, inside an expert the
    // highest ordinals first) and fill f takes the range [b_f, b_f + d_f) of
    // its giver's sequence, b_f being what that giver gave before.  Every
    // (fill, expert) pair then yields its piece independently.
    const int lane = tid & 31, warp = tid >> 5, nwarp = nt >> 5;
    const unsigned full = 0xffffffffu;
    for (int h = tid; h < d.R; h += nt) {
      sGiven[h] = 0;
      sNr[h] = 0;
    }
    __syncthreads();
    if (tid < 32) {
      int nfill = 0;
      bool ok = true;
      while (true) {
        int u = -1, o = -1;
        for (int h0 = 0; h0 < d.R && (u < 0 || o < 0); h0 += 32) {
          const int h = h0 + lane;
          const int st = h < d.R ? sState[h] : kBalanced;
          const unsigned mu = __ballot_sync(full, st == kUnder), mo = __ballot_sync(full, st == kOver);
          if (u < 0 && mu) u = h0 + __ffs(mu) - 1;
          if (o < 0 && mo) o = h0 + __ffs(mo) - 1;
        }
        if (u < 0) break;
        if (o < 0 || nfill >= d.R - 1) { ok = false; break; }
        const int dcopies = d.C - sLoad[u];
        if (lane == 0) {
          sFU[nfill] = u;
          sFO[nfill] = o;
          sFD[nfill] = dcopies;
          sFB[nfill] = sGiven[o];
          sFS[nfill] = 0;
          sGiven[o] += dcopies;
          sLoad[u] = d.C;
          sState[u] = kBalanced;
          sLoad[o] -= dcopies;
          sState[o] = sLoad[o] < d.C ? kUnder : (sLoad[o] > d.C ? kOver : kBalanced);
        }
        __syncwarp();
        ++nfill;
      }
      if (lane == 0) {
        if (!ok) set_error(p.status, MOONEP_ERR_INTERNAL);
        p.counters[MOONEP_CNT_FILLS] = nfill;
        sFZ[d.R - 1] = nfill;  // the fill count, read back below (fills < R)
      }
    }
    __syncthreads();
    if (plan_failed(p.status)) return;
    const int F = sFZ[d.R - 1];
    __syncthreads();
    if (F > 0) {
      // per giver: offsets and non-empty counts of the higher-id experts
      for (int h = warp; h < d.R; h += nwarp) {
        if (sGiven[h] == 0) continue;
        int run = 0, runz = 0;
        for (int top = (h + 1) * d.L - 1; top >= h * d.L; top -= 32) {
          const int e = top - lane;
          const int v = (e >= h * d.L) ? sT[e] : 0;
          const int z = v > 0 ? 1 : 0;
          int iv = v, iz = z;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int a = __shfl_up_sync(full, iv, off), b = __shfl_up_sync(full, iz, off);
            if (lane >= off) { iv += a; iz += b; }
          }
          if (e >= h * d.L) {
            sOff[e] = run + iv - v;
            sNz[e] = runz + iz - z;
          }
          run += __shfl_sync(full, iv, 31);
          runz += __shfl_sync(full, iz, 31);
        }
      }
      __syncthreads();
      // per fill: the giver's non-empty experts used up before it
      for (int f = warp; f < F; f += nwarp) {
        const int o = sFO[f], b = sFB[f];
        int z = 0;
        for (int e = o * d.L + lane; e < (o + 1) * d.L; e += 32) {
          const int v = sT[e];
          z += (v > 0 && sOff[e] + v <= b) ? 1 : 0;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(full, z, off);
        if (lane == 0) sFZ[f] = z;
      }
      __syncthreads();
      // every (fill, giver expert) pair with copies in the fill's range
      for (int it = tid; it < F * d.L; it += nt) {
        const int f = it / d.L, i = it % d.L;
        const int o = sFO[f], u = sFU[f], b = sFB[f], dd = sFD[f];
        const int e = (o + 1) * d.L - 1 - i;
        const int te = sT[e], off = sOff[e];
        const int t = min(b + dd, off + te) - max(b, off);
        if (t <= 0) continue;
        const int left = te - max(0, b - off);  // copies of e not yet taken
        const int j = sNz[e] - sFZ[f];          // acquisition order within the fill
        int pi = 0;                             // earlier fills of this giver that took from e
        for (int f2 = 0; f2 < f; ++f2) pi += (sFO[f2] == o && sFB[f2] + sFD[f2] > off) ? 1 : 0;
        if (pi >= d.R) { set_error(p.status, MOONEP_ERR_INTERNAL); continue; }
        const int g = (j < d.B) ? d.E + j : e;
        if (j < d.B) p.slot_expert[u * d.B + j] = e;
        p.pieces[(size_t)e * d.R + pi] = Piece{left - t, left, u, g};
        atomicAdd(&sPieceN[e], 1);
        atomicAdd(&sMig[e], t);
        atomicAdd(&sFS[f], t);
        atomicAdd(&sNr[u], 1);
        p.cu[(size_t)u * (EB + 1) + g + 1] = t;
        count_group(u, t);
      }
      __syncthreads();
      for (int f = tid; f < F; f += nt) {
        const int u = sFU[f];
        p.fills[3 * f + 0] = u;
        p.fills[3 * f + 1] = sFO[f];
        p.fills[3 * f + 2] = sFD[f];
        p.src[u] = sFO[f];
        p.n_recv[u] = sNr[u];
        if (sFS[f] != sFD[f] || (d.mode == 0 && sNr[u] > d.B)) set_error(p.status, MOONEP_ERR_INTERNAL);
      }
    }
  }

  // the fills, sequential by construction (at most R-1 of them); warp 0 runs
  // them, each decision made with ballots / shuffles so all lanes agree
  if (!parallel_fills && tid < 32) {
    const int lane = tid;
    const unsigned full = 0xffffffffu;
    int nfill = 0;
    bool ok = true;
    // record one migrated range: ordinals [left - t, left) of expert e go to
    // u as its j-th acquired expert (a slot, or the home row when j >= B)
    auto emit = [&](int u, int e, int left, int t, int j) -> bool {
      const int g = (j < d.B) ? d.E + j : e;
      if (j < d.B) p.slot_expert[u * d.B + j] = e;
      const int pi = sPieceN[e];
      if (pi >= d.R) return false;
      p.pieces[(size_t)e * d.R + pi] = Piece{left - t, left, u, g};
      sPieceN[e] = pi + 1;
      p.cu[(size_t)u * (EB + 1) + g + 1] = t;
      count_group(u, t);
      sMig[e] += t;
      return true;
    };
    while (ok) {
      int u = -1, o = -1;
      if (d.policy == 1) {
        // largest deficit / largest surplus, ties to the smallest id: per-lane
        // best over a strided subset, then a warp argmax
        int bd = 0, bs = 0;
        for (int h = lane; h < d.R; h += 32) {
          const int st = sState[h], ld = sLoad[h];
          if (st == kUnder && d.C - ld > bd) { bd = d.C - ld; u = h; }
          if (st == kOver && ld - d.C > bs) { bs = ld - d.C; o = h; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const int od = __shfl_xor_sync(full, bd, off), ou = __shfl_xor_sync(full, u, off);
          if (ou >= 0 && (u < 0 || od > bd || (od == bd && ou < u))) { bd = od; u = ou; }
          const int os = __shfl_xor_sync(full, bs, off), oo = __shfl_xor_sync(full, o, off);
          if (oo >= 0 && (o < 0 || os > bs || (os == bs && oo < o))) { bs = os; o = oo; }
        }
      } else {
        // the smallest-id underloaded and overloaded ranks
        for (int h0 = 0; h0 < d.R && (u < 0 || o < 0); h0 += 32) {
          const int h = h0 + lane;
          const int st = h < d.R ? sState[h] : kBalanced;
          const unsigned mu = __ballot_sync(full, st == kUnder), mo = __ballot_sync(full, st == kOver);
          if (u < 0 && mu) u = h0 + __ffs(mu) - 1;
          if (o < 0 && mo) o = h0 + __ffs(mo) - 1;
        }
      }
      if (u < 0) break;
      if (o < 0 || nfill >= d.R - 1) { ok = false; break; }
      const int dcopies = d.C - sLoad[u];
      int need = dcopies, j = 0;
      if (d.policy == 1) {
        // repeatedly the donor expert with the most copies left, ties to the highest id
        while (need > 0 && ok) {
          int bl = 0, be = -1;
          for (int c = o * d.L + lane; c < (o + 1) * d.L; c += 32) {
            const int lc = sT[c] - sMig[c];
            if (lc > 0 && lc >= bl) { bl = lc; be = c; }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const int ol = __shfl_xor_sync(full, bl, off), oe = __shfl_xor_sync(full, be, off);
            if (ol > bl || (ol == bl && oe > be)) { bl = ol; be = oe; }
          }
          if (be < 0) { ok = false; break; }
          const int t = min(bl, need);
          bool good = true;
          if (lane == 0) good = emit(u, be, bl, t, j);
          ok = __shfl_sync(full, good, 0);
          __syncwarp();
          need -= t;
          ++j;
        }
      } else {
        // o's experts in descending id, 32 at a time: each takes min(left,
        // what is still needed after the higher ones)
        for (int top = (o + 1) * d.L - 1; top >= o * d.L && need > 0 && ok; top -= 32) {
          const int e = top - lane;
          const int left = (e >= o * d.L) ? sT[e] - sMig[e] : 0;
          int incl = left;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(full, incl, off);
            if (lane >= off) incl += v;
          }
          const int t = max(0, min(left, need - (incl - left)));
          const unsigned mt = __ballot_sync(full, t > 0);
          bool good = true;
          if (t > 0) good = emit(u, e, left, t, j + __popc(mt & ((1u << lane) - 1u)));
          ok = __all_sync(full, good);
          __syncwarp();
          j += __popc(mt);
          need -= min(need, __shfl_sync(full, incl, 31));
        }
        if (need > 0) ok = false;  // o ran out of copies (cannot happen for an overloaded o)
      }
      if (!ok) break;
      if (d.mode == 0 && j > d.B) { ok = false; break; }
      if (lane == 0) {
        p.fills[3 * nfill + 0] = u;
        p.fills[3 * nfill + 1] = o;
        p.fills[3 * nfill + 2] = dcopies;
        p.n_recv[u] = j;
        p.src[u] = o;
        sLoad[u] = d.C;
        sState[u] = kBalanced;
        sLoad[o] -= dcopies;
        sState[o] = sLoad[o] < d.C ? kUnder : (sLoad[o] > d.C ? kOver : kBalanced);
      }
      __syncwarp();
      ++nfill;
    }
    if (lane == 0) {
      if (!ok) set_error(p.status, MOONEP_ERR_INTERNAL);
      p.counters[MOONEP_CNT_FILLS] = nfill;
    }
  }
  __syncthreads();
  if (plan_failed(p.status)) return;

  // keep, home rows, per-rank tile counts
  for (int e = tid; e < d.E; e += nt) {
    p.piece_n[e] = sPieceN[e];
    const int k = sT[e] - sMig[e];
    p.keep[e] = k;
    const int h = e / d.L;
    p.cu[(size_t)h * (EB + 1) + e + 1] = k;
    if (k > 0) count_group(h, k);
  }
  // reduce lists: the slots holding e in ascending (u, j)
  for (int s = tid; s < d.R * d.B; s += nt) {
    const int e = p.slot_expert[s];
    if (e >= 0) {
      const int at = atomicAdd(&p.red_n[e], 1);
      p.red_slots[(size_t)e * d.R + at] = s;
    }
  }
  __syncthreads();
  for (int e = tid; e < d.E; e += nt) {
    const int n = p.red_n[e];
    int32_t* l = p.red_slots + (size_t)e * d.R;
    for (int a = 1; a < n; ++a) {  // insertion sort, n <= R-1
      const int v = l[a];
      int b = a - 1;
      while (b >= 0 && l[b] > v) { l[b + 1] = l[b]; --b; }
      l[b + 1] = v;
    }
  }
  // compact lists (warp 0, ballot prefix keeps ascending order)
  if (tid < 32) {
    int n_occ = 0, n_red = 0;
    for (int s0 = 0; s0 < d.R * d.B; s0 += 32) {
      const int s = s0 + tid;
      const bool occ = s < d.R * d.B && p.slot_expert[s] >= 0;
      const unsigned m = __ballot_sync(0xffffffffu, occ);
      if (occ) p.occupied[n_occ + __popc(m & ((1u << tid) - 1u))] = s;
      n_occ += __popc(m);
    }
    for (int e0 = 0; e0 < d.E; e0 += 32) {
      const int e = e0 + tid;
      const bool has = e < d.E && p.red_n[e] > 0;
      const unsigned m = __ballot_sync(0xffffffffu, has);
      if (has) p.red_list[n_red + __popc(m & ((1u << tid) - 1u))] = e;
      n_red += __popc(m);
    }
    if (tid == 0) {
      p.counters[MOONEP_CNT_OCCUPIED] = n_occ;
      p.counters[MOONEP_CNT_REDUCE] = n_red;
      // the GEMMs' work-tile height: fixed by the dims, or the cheaper one
      // under the cost model for this plan's group sizes
      long long n128 = 0, n256f = 0, n256h = 0, ng = 0;
      for (int h = 0; h < d.R; ++h) {
        n128 += sT128[h];
        n256f += sT256F[h];
        n256h += sT256H[h];
        ng += sGroups[h];
      }
      const int rows = d.tile_m ? d.tile_m : gemm_tile_rows_for(n128, n256f, n256h, ng, d.Hp);
      p.counters[MOONEP_CNT_TILE_ROWS] = rows;
      int run = 0;
      for (int h = 0; h < d.R; ++h) {
        p.rank_tiles[h] = run;
        run += (rows == kMmaM) ? sT128[h] : sT256F[h] + sT256H[h];
      }
      p.rank_tiles[d.R] = run;
      p.counters[MOONEP_CNT_MTILES] = run;
      if (run > d.max_mtiles) set_error(p.status, MOONEP_ERR_INTERNAL);
      run = 0;
      for (int h = 0; h < d.R; ++h) {
        p.rank_groups[h] = run;
        run += sGroups[h];
      }
      p.rank_groups[d.R] = run;
      p.counters[MOONEP_CNT_GROUPS] = run;
      if (run > d.max_groups) set_error(p.status, MOONEP_ERR_INTERNAL);
    }
  }
}

// ---------------------------------------------------------------------------
// 3. per-rank tables: cu_seqlens scan, GEMM tile list, row bases
//    grid R, 1024 threads
// ---------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void block_scan3(int& a, int& b, int& c, int* sa, int* sb, int* sc) {
  // inclusive block scan of three ints; sa/sb/sc hold NT/32 partials each
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, a, o);
    const int yb = __shfl_up_sync(0xffffffffu, b, o);
    const int yc = __shfl_up_sync(0xffffffffu, c, o);
    if (lane >= o) { a += ya; b += yb; c += yc; }
  }
  if (lane == 31) { sa[warp] = a; sb[warp] = b; sc[warp] = c; }
  __syncthreads();
  if (warp == 0) {
    int xa = lane < NT / 32 ? sa[lane] : 0, xb = lane < NT / 32 ? sb[lane] : 0;
    int xc = lane < NT / 32 ? sc[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, xa, o);
      const int yb = __shfl_up_sync(0xffffffffu, xb, o);
      const int yc = __shfl_up_sync(0xffffffffu, xc, o);
      if (lane >= o) { xa += ya; xb += yb; xc += yc; }
    }
    if (lane < NT / 32) { sa[lane] = xa; sb[lane] = xb; sc[lane] = xc; }
  }
  __syncthreads();
  if (warp > 0) { a += sa[warp - 1]; b += sb[warp - 1]; c += sc[warp - 1]; }
}

__global__ void __launch_bounds__(1024)
k_tables(Dims d, PlanPtrs p) {
  __shared__ int sa[32], sb[32], sc[32];
  if (plan_failed(p.status)) return;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int EB = d.E + d.B;
  int32_t* cu = p.cu + (size_t)u * (EB + 1);
  // each thread scans a contiguous run of groups
  const int per = (EB + 1023) / 1024;
  const int g0 = min(EB, tid * per), g1 = min(EB, g0 + per);
  const int tile_m = p.counters[MOONEP_CNT_TILE_ROWS];
  int rows_local[8];
  int rsum = 0, tsum = 0, gsum = 0;
  for (int g = g0, i = 0; g < g1; ++g, ++i) {
    const int rows = cu[g + 1];
    if (i < 8) rows_local[i] = rows;
    rsum += rows;
    tsum += (rows + tile_m - 1) / tile_m;
    gsum += rows > 0;
  }
  int ra = rsum, tb = tsum, gc = gsum;
  block_scan3<1024>(ra, tb, gc, sa, sb, sc);
  int row = ra - rsum, tile = tb - tsum + p.rank_tiles[u], grp = gc - gsum + p.rank_groups[u];
  __syncthreads();  // every thread has read its rows before they are replaced
  for (int g = g0, i = 0; g < g1; ++g, ++i) {
    const int rows = (i < 8) ? rows_local[i] : 0;  // per <= 8: E + B <= 2 * 4096
    cu[g] = row;
    const int wsel = (g < d.E) ? g : -1 - (u * d.B + (g - d.E));
    for (int m = 0; m * tile_m < rows; ++m) {
      p.mtiles[tile++] = MTile{u * d.C + row + m * tile_m, min(tile_m, rows - m * tile_m), wsel, u};
    }
    if (rows > 0) p.groups[grp++] = MTile{u * d.C + row, rows, wsel, u};
    row += rows;
  }
  if (tid == 1023) cu[EB] = row;
  __syncthreads();
  // row bases: home experts of u, and every piece that lands on u
  for (int e = u * d.L + tid; e < (u + 1) * d.L; e += 1024) p.home_base[e] = u * d.C + cu[e];
  for (int e = tid; e < d.E; e += 1024) {
    const int n = p.piece_n[e];
    for (int i = 0; i < n; ++i) {
      const Piece pc = p.pieces[(size_t)e * d.R + i];
      if (pc.u == u) p.piece_base[(size_t)e * d.R + i] = u * d.C + cu[pc.g] - pc.lo;
    }
  }
}

// ---------------------------------------------------------------------------
// 4. destinations and inverse: grid (nchunk * kDstSplit, R), 256 threads;
//    the kDstSplit CTAs of a chunk interleave its copies, so each thread
//    follows at most four copies' chains of dependent loads
// ---------------------------------------------------------------------------
constexpr int kDstSplit = 4;

__global__ void __launch_bounds__(256)
k_dst(Dims d, const int32_t* __restrict__ idx, PlanPtrs p) {
  if (plan_failed(p.status)) return;
  const int r = blockIdx.y, chunk = blockIdx.x / kDstSplit, part = blockIdx.x % kDstSplit;
  const int t0 = chunk * d.chunk_tokens;
  const int t1 = min(d.S, t0 + d.chunk_tokens);
  const int ncopy = (t1 - t0) * d.K;
  const size_t first = ((size_t)r * d.S + t0) * d.K;
  const int32_t* base = p.counts + ((size_t)r * d.nchunk + chunk) * d.E;
  for (int i = part * blockDim.x + threadIdx.x; i < ncopy; i += kDstSplit * blockDim.x) {
    const size_t c = first + i;
    const int e = idx[c];
    const int q = base[e] + p.gidx[c];
    p.gidx[c] = q;
    int row;
    if (q < p.keep[e]) {
      row = p.home_base[e] + q;
    } else {
      row = -1;
      const int n = p.piece_n[e];
      for (int j = 0; j < n; ++j) {
        const Piece pc = p.pieces[(size_t)e * d.R + j];
        if (pc.lo <= q && q < pc.hi) { row = p.piece_base[(size_t)e * d.R + j] + q; break; }
      }
      if (row < 0) { set_error(p.status, MOONEP_ERR_INTERNAL); continue; }
    }
    if (row < 0 || row >= d.N) { set_error(p.status, MOONEP_ERR_INTERNAL); continue; }
    p.dst[c] = row;
    p.inverse[row] = (int32_t)c;
  }
}

// ---------------------------------------------------------------------------
// 5. send-once route entries ("Kimi K3 模型结构（8）", section 在线规划、零拷贝、
//    静态 shape): per token, entry k keeps its row offset on its destination
//    rank unless an earlier entry of the token goes to the same rank, in which
//    case it stores -offset-1.  Also counts the entries and the distinct
//    (token, rank) pairs that leave the token's own rank.  One thread per token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_route(Dims d, PlanPtrs p) {
  if (plan_failed(p.status)) return;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  int entries = 0, pairs = 0;
  if (t < d.R * d.S) {
    const int r = t / d.S;
    const int32_t* dt = p.dst + (size_t)t * d.K;
    int32_t* rt = p.route + (size_t)t * d.K;
    // destination ranks of the first kRouteRegs entries kept in registers, so
    // the earlier-entry test costs no reloads or divisions
    constexpr int kRouteRegs = 32;
    int ur[kRouteRegs];
#pragma unroll
    for (int j = 0; j < kRouteRegs; ++j) ur[j] = -1;
    for (int k = 0; k < d.K; ++k) {
      const int v = dt[k];
      const int u = v / d.C;
      bool dup = false;
      if (k <= kRouteRegs) {
#pragma unroll
        for (int j = 0; j < kRouteRegs; ++j) dup |= (j < k) && (ur[j] == u);
      } else {
#pragma unroll
        for (int j = 0; j < kRouteRegs; ++j) dup |= (ur[j] == u);
        for (int j = kRouteRegs; j < k; ++j) dup |= (dt[j] / d.C == u);
      }
#pragma unroll
      for (int j = 0; j < kRouteRegs; ++j) ur[j] = (j == k) ? u : ur[j];
      const int off = v - u * d.C;
      rt[k] = dup ? -off - 1 : off;
      if (u != r) {
        ++entries;
        pairs += dup ? 0 : 1;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    entries += __shfl_xor_sync(0xffffffffu, entries, o);
    pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
  }
  if ((threadIdx.x & 31) == 0 && (entries | pairs)) {
    atomicAdd(&p.counters[MOONEP_CNT_REMOTE_ENTRIES], entries);
    atomicAdd(&p.counters[MOONEP_CNT_REMOTE_PAIRS], pairs);
  }
}

cudaError_t launch_plan(const Dims& d, const int32_t* idx, const PlanPtrs& p, cudaStream_t st,
                        int* launches) {
  cudaError_t err = cudaMemsetAsync(p.status, 0, 256, st);  // status + counters header
  if (err != cudaSuccess) return err;
  const size_t hist_smem = sizeof(int32_t) * kHistWarps * d.E;
  if (hist_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(k_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_smem);
    if (err != cudaSuccess) return err;
  }
  k_hist<<<dim3(d.nchunk, d.R), kHistWarps * 32, hist_smem, st>>>(d, idx, p);
  const size_t plan_smem = plan_smem_bytes(d);
  if (plan_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(k_plan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_smem);
    if (err != cudaSuccess) return err;
  }
  k_scan<<<(d.E + 31) / 32, 1024, 0, st>>>(d, p);
  k_plan<<<1, 1024, plan_smem, st>>>(d, p);
  k_tables<<<d.R, 1024, 0, st>>>(d, p);
  k_dst<<<dim3(d.nchunk * kDstSplit, d.R), 256, 0, st>>>(d, idx, p);
  k_route<<<(d.R * d.S + 255) / 256, 256, 0, st>>>(d, p);
  *launches += 6;
  return cudaGetLastError();
}

}  // namespace moonep
