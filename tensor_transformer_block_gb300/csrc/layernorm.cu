// LayerNorm over the hidden dimension of bf16 rows (zouht 张量并行 §2.2.2:
// mu = mean(h_i), sigma^2 = mean((h_i - mu)^2), h_hat = (h - mu) / sqrt(sigma^2 + eps),
// h' = gamma * h_hat + beta), its backward with an optional residual gradient
// added in, and the fixed-order column sums that finish dgamma and dbeta.
//
// Both row kernels are HBM-bound: every element is read once and written once.
// A row is held in registers by one CTA: thread t owns the 16-byte vectors t,
// t + blockDim, ... (VPT of them), so the loads of a warp are contiguous 512-byte
// runs.  The forward is persistent over rows and loads the next row while it
// reduces the current one, so that every SM keeps a row's worth of loads in
// flight; from h = 4096 up it takes four vectors per thread (h = 8192: 256 threads,
// four CTAs per SM), below that one.  The backward, which also keeps dgamma /
// dbeta partials per thread, loads a row's dR together with X and dY and the
// next row while it reduces the current one, with at most 512 threads (two
// vectors per thread from h = 4096 up); above h = 8192 a row needs more threads
// than those registers allow, and it loads row by row.
// Statistics are fp32, taken in two passes over the registers (mean first,
// then the centred sum of squares), so no cancellation.
//
// The backward is persistent over rows: CTA b takes rows b, b + grid, ... and,
// because each thread always owns the same columns, accumulates its columns'
// dgamma / dbeta partial sums in registers; each CTA writes one partial row and
// k_ln_colsum adds the partial rows in a fixed order.  Both kernels' launch
// geometry depends only on T, h and the device (the grids are the CTAs that fit
// at once), so the result is bit-reproducible on a given GPU.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "host_util.cuh"
#include "ln.cuh"
#include "ptx.cuh"

namespace tpb {
namespace {

// Eight 16-bit values of a 16-byte vector, bf16 or (f16) fp16, to fp32 and back.
__device__ __forceinline__ void unpack8(const uint4& q, float (&v)[8], bool f16 = false) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (f16) {
      const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      v[2 * e] = t.x;
      v[2 * e + 1] = t.y;
    } else {
      v[2 * e] = bf16lo_to_f32(w[e]);
      v[2 * e + 1] = bf16hi_to_f32(w[e]);
    }
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8], bool f16 = false) {
  uint4 q;
  q.x = f16 ? pack_f16x2(v[0], v[1]) : pack_bf16x2(v[0], v[1]);
  q.y = f16 ? pack_f16x2(v[2], v[3]) : pack_bf16x2(v[2], v[3]);
  q.z = f16 ? pack_f16x2(v[4], v[5]) : pack_bf16x2(v[4], v[5]);
  q.w = f16 ? pack_f16x2(v[6], v[7]) : pack_bf16x2(v[6], v[7]);
  return q;
}

// Sum of one value (or two) over the CTA; every thread gets the result.
// ``red`` holds 2 x 32 floats; the leading barrier protects its previous use.
__device__ __forceinline__ float2 block_sum2(float a, float b, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if (lane == 0) {
    red[warp] = a;
    red[32 + warp] = b;
  }
  __syncthreads();
  a = lane < nw ? red[lane] : 0.0f;
  b = lane < nw ? red[32 + lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  return make_float2(a, b);
}

template <int VPT>
__global__ void __launch_bounds__(1024) k_ln_fwd(const uint4* __restrict__ X, const uint4* __restrict__ gamma,
                                                 const uint4* __restrict__ beta, uint4* __restrict__ Y,
                                                 float* __restrict__ mean, float* __restrict__ rstd, int T,
                                                 int nvec, float inv_h, float eps, int io, unsigned* err) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  __shared__ float red[64];
  const bool x16 = io & kLnXF16, y16 = io & kLnYF16;
  int64_t row = blockIdx.x;
  if (row >= T) return;
  // persistent over rows: the next row's vectors are loaded while this one is reduced
  uint4 cur[VPT], nxt[VPT];
  auto load = [&](int64_t r, uint4 (&q)[VPT]) {
    const uint4* xr = X + r * nvec;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      q[k] = i < nvec ? xr[i] : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load(row, cur);
  for (; row < T; row += gridDim.x) {
    const int64_t nrow = row + gridDim.x;
    if (nrow < T) load(nrow, nxt);
    float v[VPT][8];
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      unpack8(cur[k], v[k], x16);  // zero beyond the row: adds nothing
#pragma unroll
      for (int e = 0; e < 8; ++e) s += v[k][e];
    }
    const float mu = block_sum2(s, 0.0f, red).x * inv_h;
    float q = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (threadIdx.x + k * blockDim.x < nvec) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dlt = v[k][e] - mu;
          q = fmaf(dlt, dlt, q);
        }
      }
    }
    const float var = block_sum2(q, 0.0f, red).x * inv_h;
    const float r = rsqrtf(var + eps);
    uint4* yr = Y + row * nvec;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < nvec && TP_DCHECK(row * nvec + i < static_cast<int64_t>(T) * nvec, err)) {
        float g[8], b[8], o[8];
        unpack8(gamma[i], g);
        unpack8(beta[i], b);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf((v[k][e] - mu) * r, g[e], b[e]);
        yr[i] = pack8(o, y16);
      }
    }
    if (threadIdx.x == 0) {
      mean[row] = mu;
      rstd[row] = r;
    }
#pragma unroll
    for (int k = 0; k < VPT; ++k) cur[k] = nxt[k];
  }
}

// PF: the row's dR is loaded with X and dY, and the next row's three vectors are
// loaded while this row is reduced (more registers: at most 512 threads).
template <int VPT, bool PF>
__global__ void __launch_bounds__(PF ? 512 : 1024)
    k_ln_bwd(const uint4* __restrict__ X, const uint4* __restrict__ gamma, const float* __restrict__ mean,
             const float* __restrict__ rstd, const uint4* __restrict__ dY, const uint4* __restrict__ dR,
             uint4* __restrict__ dX, float* __restrict__ part, int T, int nvec, float inv_h, int io,
             unsigned* err) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  __shared__ float red[64];
  const bool x16 = io & kLnXF16, dy16 = io & kLnDyF16, dr16 = io & kLnDrF16, dx16 = io & kLnDxF16;
  float gm[VPT][8], pg[VPT][8], pb[VPT][8];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < nvec) {
      unpack8(gamma[i], gm[k]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) gm[k][e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pg[k][e] = 0.0f;
      pb[k][e] = 0.0f;
    }
  }
  // raw vectors of X, dY, dR for one row (zero past the row, or dR absent)
  struct RowIn {
    uint4 x[VPT], dy[VPT], dr[VPT];
  };
  auto load = [&](int64_t row, RowIn& q) {
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      const bool in = i < nvec;
      q.x[k] = in ? X[row * nvec + i] : make_uint4(0u, 0u, 0u, 0u);
      q.dy[k] = in ? dY[row * nvec + i] : make_uint4(0u, 0u, 0u, 0u);
      if (PF) q.dr[k] = (in && dR) ? dR[row * nvec + i] : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  RowIn cur, nxt;
  if (PF && blockIdx.x < T) load(blockIdx.x, cur);
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    if (PF) {
      if (row + gridDim.x < T) load(row + gridDim.x, nxt);
    } else {
      load(row, cur);
    }
    const float mu = mean[row], r = rstd[row];
    float xh[VPT][8], g[VPT][8];
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < nvec) {
        float xv[8], dy[8];
        unpack8(cur.x[k], xv, x16);
        unpack8(cur.dy[k], dy, dy16);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xh[k][e] = (xv[e] - mu) * r;
          g[k][e] = dy[e] * gm[k][e];
          s1 += g[k][e];
          s2 = fmaf(g[k][e], xh[k][e], s2);
          pg[k][e] = fmaf(dy[e], xh[k][e], pg[k][e]);
          pb[k][e] += dy[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          xh[k][e] = 0.0f;
          g[k][e] = 0.0f;
        }
      }
    }
    const float2 c = block_sum2(s1, s2, red);
    const float c1 = c.x * inv_h, c2 = c.y * inv_h;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < nvec && TP_DCHECK(row * nvec + i < static_cast<int64_t>(T) * nvec, err)) {
        float o[8], rr[8];
        // zero without a residual (without the prefetch, loaded only now)
        unpack8(PF ? cur.dr[k] : (dR ? dR[row * nvec + i] : make_uint4(0u, 0u, 0u, 0u)), rr, dr16);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = r * (g[k][e] - c1 - xh[k][e] * c2) + rr[e];
        dX[row * nvec + i] = pack8(o, dx16);
      }
    }
    if (PF) cur = nxt;
  }
  // partial row of this CTA: [2][h] fp32 (dgamma, then dbeta)
  float* pr = part + static_cast<int64_t>(blockIdx.x) * 2 * nvec * 8;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < nvec) {
      float4* a = reinterpret_cast<float4*>(pr + i * 8);
      float4* b = reinterpret_cast<float4*>(pr + nvec * 8 + i * 8);
      a[0] = make_float4(pg[k][0], pg[k][1], pg[k][2], pg[k][3]);
      a[1] = make_float4(pg[k][4], pg[k][5], pg[k][6], pg[k][7]);
      b[0] = make_float4(pb[k][0], pb[k][1], pb[k][2], pb[k][3]);
      b[1] = make_float4(pb[k][4], pb[k][5], pb[k][6], pb[k][7]);
    }
  }
}

// out[c] = bf16(sum_{p=0}^{P-1} part[p][c]) for c < 2h (dgamma then dbeta).  A CTA
// of 8 warps takes 32 columns: warp w adds rows w, w + 8, ... in order, then lane c
// of warp 0 adds the 8 warp sums in order, so the sum's order is fixed by P alone.
constexpr int kColsumWarps = 8;
__global__ void __launch_bounds__(kColsumWarps * 32) k_ln_colsum(const float* __restrict__ part, int P, int two_h,
                                                                   int h, __nv_bfloat16* dgamma,
                                                                   __nv_bfloat16* dbeta) {
  grid_dep_wait();  // the previous kernel in the stream has completed
  grid_dep_launch();
  __shared__ float red[kColsumWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (c < two_h) {
#pragma unroll 4
    for (int p = warp; p < P; p += kColsumWarps) s += part[static_cast<int64_t>(p) * two_h + c];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < two_h) {
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kColsumWarps; ++w) t += red[w][lane];
    if (c < h)
      dgamma[c] = __float2bfloat16_rn(t);
    else
      dbeta[c - h] = __float2bfloat16_rn(t);
  }
}

struct LnGeom {
  int vpt, threads;
  bool pf = false;  // backward: dR with X and dY, next row prefetched
};

// forward: four vectors per thread from h = 4096 up (fewer threads per row, more
// rows per SM), one below (a narrow row would leave a CTA one warp wide)
LnGeom ln_fwd_geom(int64_t h) {
  const int64_t nvec = h / 8;
  LnGeom g{nvec >= 512 ? 4 : 1, 32};
  const int64_t t = (nvec + g.vpt - 1) / g.vpt;
  g.threads = static_cast<int>((t + 31) / 32 * 32);
  return g;
}

// backward: up to h = 8192 the prefetching kernel with at most 512 threads (two
// vectors per thread from h = 4096 up); above that two vectors per thread, no
// prefetch (a row then needs up to 1024 threads, whose registers leave no room)
LnGeom ln_geom(int64_t h) {
  const int64_t nvec = h / 8;
  LnGeom g{1, 32};
  g.pf = nvec <= 1024;
  g.vpt = g.pf ? (nvec >= 512 ? 2 : 1) : 2;
  const int64_t t = (nvec + g.vpt - 1) / g.vpt;
  g.threads = static_cast<int>((t + 31) / 32 * 32);
  return g;
}

int ln_bwd_grid(int64_t T, int threads) {
  const int sms = device_sm_count();
  const int per_sm = threads > 0 ? 2048 / threads : 1;
  int64_t g = static_cast<int64_t>(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
  if (g > T) g = T;
  return static_cast<int>(g);
}

}  // namespace

bool ln_shape_ok(int64_t T, int64_t h) { return T >= 1 && h >= 8 && h % 8 == 0 && h <= kLnMaxH && T < (1ll << 31); }

size_t ln_partial_bytes(int64_t T, int64_t h) {
  const LnGeom g = ln_geom(h);
  return static_cast<size_t>(ln_bwd_grid(T, g.threads)) * 2 * static_cast<size_t>(h) * sizeof(float);
}

int launch_ln_fwd(const void* X, const void* gamma, const void* beta, void* Y, float* mean, float* rstd, int64_t T,
                  int64_t h, float eps, cudaStream_t st, int io, unsigned* err) {
  if (!ln_shape_ok(T, h)) return 1;
  const LnGeom g = ln_fwd_geom(h);
  const int nvec = static_cast<int>(h / 8);
  const float inv_h = 1.0f / static_cast<float>(h);
  const auto* x = static_cast<const uint4*>(X);
  const auto* ga = static_cast<const uint4*>(gamma);
  const auto* be = static_cast<const uint4*>(beta);
  auto* y = static_cast<uint4*>(Y);
  // resident CTAs per SM for this shape (the grid is what fits at once)
  int per_sm = 0;
  const cudaError_t oe = g.vpt == 4
                             ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_fwd<4>, g.threads, 0)
                             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_fwd<1>, g.threads, 0);
  if (oe != cudaSuccess) return 2;
  int64_t nb = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
  if (nb > T) nb = T;
  const int slot = timing_begin(kKLnFwd, st);
  const dim3 grid(static_cast<unsigned>(nb));
  const bool ok = launch_k(g.vpt == 4 ? k_ln_fwd<4> : k_ln_fwd<1>, grid, dim3(g.threads), 0, st, 1, x, ga, be, y,
                           mean, rstd, static_cast<int>(T), nvec, inv_h, eps, io, err) == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

int launch_ln_bwd(const void* X, const void* gamma, const float* mean, const float* rstd, const void* dY,
                  const void* dR, void* dX, void* dgamma, void* dbeta, float* part, int64_t T, int64_t h,
                  cudaStream_t st, int io, unsigned* err) {
  if (!ln_shape_ok(T, h)) return 1;
  const LnGeom g = ln_geom(h);
  const int nvec = static_cast<int>(h / 8);
  const float inv_h = 1.0f / static_cast<float>(h);
  // as many persistent CTAs as fit at once (never more than the partials allow)
  int per_sm = 0;
  cudaError_t oe;
  if (g.pf)
    oe = g.vpt == 2 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_bwd<2, true>, g.threads, 0)
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_bwd<1, true>, g.threads, 0);
  else
    oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ln_bwd<2, false>, g.threads, 0);
  if (oe != cudaSuccess) return 2;
  int grid = ln_bwd_grid(T, g.threads);
  const int64_t fit = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
  if (fit < grid) grid = static_cast<int>(fit);
  const auto* x = static_cast<const uint4*>(X);
  const auto* ga = static_cast<const uint4*>(gamma);
  const auto* dy = static_cast<const uint4*>(dY);
  const auto* dr = static_cast<const uint4*>(dR);
  auto* dx = static_cast<uint4*>(dX);
  int slot = timing_begin(kKLnBwd, st);
  bool ok = launch_k(g.pf ? (g.vpt == 2 ? k_ln_bwd<2, true> : k_ln_bwd<1, true>) : k_ln_bwd<2, false>,
                     dim3(static_cast<unsigned>(grid)), dim3(g.threads), 0, st, 1, x, ga, mean, rstd, dy, dr, dx, part,
                     static_cast<int>(T), nvec, inv_h, io, err) == cudaSuccess;
  timing_end(slot, st);
  if (!ok) return 2;
  slot = timing_begin(kKLnColsum, st);
  const int two_h = static_cast<int>(2 * h);
  ok = launch_k(k_ln_colsum, dim3(static_cast<unsigned>((two_h + 31) / 32)), dim3(kColsumWarps * 32), 0, st, 1,
                static_cast<const float*>(part), grid, two_h, static_cast<int>(h),
                static_cast<__nv_bfloat16*>(dgamma), static_cast<__nv_bfloat16*>(dbeta)) == cudaSuccess;
  timing_end(slot, st);
  return ok ? 0 : 2;
}

}  // namespace tpb
