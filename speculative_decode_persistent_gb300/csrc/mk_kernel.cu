// The persistent verify-step kernel.
//
// One cooperative launch runs the whole cycle that the page "Fusing the whole
// speculative-decoding cycle into one CUDA kernel" (section "What shipped")
// describes: the main model over every row of every sequence, lm_head, greedy
// verification, all as phases of ONE launch separated by a software grid
// barrier; the host reads back only the accepted tokens.
//
// Phase order per step (every block runs every phase):
//   embed -> per layer [input GEMM | mixer (Gated DeltaNet or attention) |
//   o_proj GEMM | gate/up GEMM | down GEMM] -> lm_head GEMM -> verify.
//
// Weight streaming: every warp owns a ring of kRing 4.6 KB units filled by
// bulk asynchronous copies (cp.async.bulk + mbarrier). The GEMM schedule is
// static, so a warp keeps issuing the copies of its NEXT units — across the
// grid barrier and through the mixer phases — while it waits; HBM keeps
// streaming weights while the barrier settles.
//
// Skinny GEMM arithmetic (all rows of the step against each weight once):
// 4-bit codes become exact fp16 integers sc_j*q with one lop3 and one fused
// multiply-add per pair; the activations are split into two fp16 parts
// (high + low) so that the m16n8k16 products stay exact to ~2^-22; each
// super-block's fp16 tile sums are scaled by d in fp32 and the min term
// dmin * sum_j m_j * sum(x over sub-block j) is added by the lane that owns
// the weight row. Weights are therefore used exactly as stored.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "mk_internal.cuh"

namespace mk {

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
  return r;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float sigmoidf_(float v) { return 1.0f / (1.0f + expf(-v)); }
__device__ __forceinline__ float siluf_(float v) { return v / (1.0f + expf(-v)); }

// --------------------------------------------------------- shared memory
struct Smem {
  uint8_t* base;
  __device__ uint8_t* ring(int warp, int slot) const {
    return base + kOffRing + (warp * kRing + slot) * kUnitBytes;
  }
  __device__ uint64_t* bar(int warp, int slot) const {
    return reinterpret_cast<uint64_t*>(base + kOffBar) + warp * kRing + slot;
  }
  __device__ uint32_t* stab(int warp) const {
    return reinterpret_cast<uint32_t*>(base + kOffTab + warp * kWarpTab);
  }
  __device__ float* dtab(int warp) const {
    return reinterpret_cast<float*>(base + kOffTab + warp * kWarpTab + kScaleTab);
  }
  __device__ uint8_t* act() const { return base + kOffAct; }
  __device__ float* misc() const { return reinterpret_cast<float*>(base + kOffMisc); }
  __device__ uint8_t* phase() const { return base + kOffPhase; }
};

// -------------------------------------------------------------- grid sync
// Sense by generation: read the generation, arrive, and wait (bounded) until
// the last arriver bumps it. An error word set by any block makes every
// waiter leave at its next check; a wait that outlives the deadline sets it.
__device__ bool grid_sync(const ModelDesc& md, const StepDesc& sd, int& nbar, int* sflag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile int32_t* err = md.err;
    const uint32_t gen = ld_acquire(&md.bar[1]);
    const bool skip = sd.skip_block == static_cast<int>(blockIdx.x) && sd.skip_barrier == nbar;
    if (*err == 0 && !skip) {
      __threadfence();
      const uint32_t arrived = atomicAdd(&md.bar[0], 1u) + 1u;
      if (arrived == gridDim.x) {
        atomicExch(&md.bar[0], 0u);
        __threadfence();
        st_release(&md.bar[1], gen + 1u);
      }
    }
    const uint64_t t0 = globaltimer();
    uint32_t ns = 32;
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire(&md.bar[1]) != gen) break;
      if (*err != 0) { ok = 0; break; }
      if (globaltimer() - t0 > sd.barrier_timeout_ns || it > (1u << 28)) {
        atomicCAS(md.err, 0, DEV_BARRIER_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(ns);
      if (ns < 256) ns <<= 1;
    }
    if (*err != 0) ok = 0;
    __threadfence();
    *sflag = ok;
  }
  __syncthreads();
  ++nbar;
  return *sflag != 0;
}

// ------------------------------------------------------------ the stream
struct WarpCtx {
  int warp, lane, gid;
  uint32_t c_pos, p_pos;
  int p_gp;
  bool p_done;
  int64_t p_u, p_u1;
  int p_nsb_s, p_sb0, p_nsb;
  const uint8_t* p_w;
  uint64_t pol;
};

__device__ __forceinline__ const GemmDesc& gemm_desc(const ModelDesc& md, int gp) {
  const int l = gp >> 2, part = gp & 3;
  if (l >= md.n_layers) return md.lm;
  const LayerDesc& L = md.layer[l];
  return part == 0 ? L.in : part == 1 ? L.o : part == 2 ? L.gu : L.down;
}

struct Assign {
  Sched sc;
  int sl, nsb_s, sb0, cta0;
  int64_t Us, Ws, ws, u0, u1;
};

__device__ __forceinline__ Assign assign_for(const GemmDesc& g, int R, int grid, int cta, int warp) {
  Assign a;
  a.sc = make_sched(g.nsb, R);
  a.sl = slice_of_cta(a.sc, grid, cta);
  a.cta0 = slice_cta0(a.sc, grid, a.sl);
  const int cta1 = slice_cta0(a.sc, grid, a.sl + 1);
  a.nsb_s = slice_nsb(a.sc, g.nsb, a.sl);
  a.sb0 = slice_sb0(a.sc, a.sl);
  a.Us = static_cast<int64_t>(g.n_tiles) * a.nsb_s;
  a.Ws = static_cast<int64_t>(cta1 - a.cta0) * kWarps;
  a.ws = static_cast<int64_t>(cta - a.cta0) * kWarps + warp;
  a.u0 = warp_u0(a.Us, a.Ws, a.ws);
  a.u1 = warp_u0(a.Us, a.Ws, a.ws + 1);
  return a;
}

// Issue the bulk copies of this warp's next units until its ring is full.
__device__ void produce(WarpCtx& wc, const ModelDesc& md, const StepDesc& sd, const Smem& sm) {
  while (!wc.p_done && wc.p_pos - wc.c_pos < static_cast<uint32_t>(kRing)) {
    if (wc.p_u >= wc.p_u1) {
      ++wc.p_gp;
      if (wc.p_gp > 4 * md.n_layers) { wc.p_done = true; break; }
      const GemmDesc& g = gemm_desc(md, wc.p_gp);
      const Assign a = assign_for(g, sd.R, gridDim.x, blockIdx.x, wc.warp);
      wc.p_u = a.u0;
      wc.p_u1 = a.u1;
      wc.p_nsb_s = a.nsb_s;
      wc.p_sb0 = a.sb0;
      wc.p_nsb = g.nsb;
      wc.p_w = g.w;
      continue;
    }
    const int slot = wc.p_pos % kRing;
    if (wc.lane == 0) {
      const int64_t tile = wc.p_u / wc.p_nsb_s;
      const int sb = wc.p_sb0 + static_cast<int>(wc.p_u % wc.p_nsb_s);
      const uint8_t* src = wc.p_w + (static_cast<size_t>(tile) * wc.p_nsb + sb) * kUnitBytes;
      uint64_t* b = sm.bar(wc.warp, slot);
      mbar_arrive_expect_tx(b, kUnitBytes);
      bulk_g2s(sm.ring(wc.warp, slot), src, kUnitBytes, b, wc.pol);
    }
    ++wc.p_u;
    ++wc.p_pos;
  }
}

__device__ bool wait_unit(const WarpCtx& wc, const Smem& sm, const ModelDesc& md, uint64_t timeout_ns) {
  const int slot = wc.c_pos % kRing;
  const uint32_t parity = (wc.c_pos / kRing) & 1u;
  uint64_t* b = sm.bar(wc.warp, slot);
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if (globaltimer() - t0 > timeout_ns || it > (1u << 26)) {
      atomicCAS(md.err, 0, DEV_COPY_TIMEOUT);
      return false;
    }
  }
}

// Wait (bounded) for every copy this warp still has in flight.
__device__ void drain(WarpCtx& wc, const Smem& sm, const ModelDesc& md) {
  while (wc.c_pos < wc.p_pos) {
    wait_unit(wc, sm, md, 50000000ull);
    ++wc.c_pos;
  }
}

// ------------------------------------------------------------------ embed
__device__ void embed_phase(const ModelDesc& md, const StepDesc& sd, const WarpCtx& wc) {
  const int nsbH = md.H / 256;
  const int total = sd.R * nsbH;
  for (int it = wc.gid; it < total; it += gridDim.x * kWarps) {
    const int r = it / nsbH, sb = it % nsbH;
    const uint8_t* blk = md.embed + (static_cast<size_t>(sd.row_tok[r]) * nsbH + sb) * 144;
    const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
    const uint64_t lo64 = hdr.y | (static_cast<uint64_t>(hdr.z) << 32);
    const uint64_t mid64 = hdr.z | (static_cast<uint64_t>(hdr.w) << 32);
    const int j = wc.lane / 4;
    const int i0 = (wc.lane % 4) * 8;
    const float sc = static_cast<float>((lo64 >> (6 * j)) & 63u);
    const float m = static_cast<float>((mid64 >> (16 + 6 * j)) & 63u);
    const float ds = d * sc, dm = dmin * m;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = i0 + e;
      const uint8_t byte = __ldg(blk + 16 + 16 * j + (i % 16));
      const int q = i < 16 ? (byte & 15) : (byte >> 4);
      md.x[static_cast<size_t>(r) * md.H + sb * 256 + 32 * j + i] = ds * static_cast<float>(q) - dm;
    }
  }
}

// --------------------------------------------------------- GEMM prologue
// Fills the activation region for reduction slice [sb0, sb0 + nsb_s): for each
// row r, column 2r holds the fp16 high part and column 2r+1 the low part of the
// input vector, each column in the per-32 permuted order of the B fragments;
// then sx[sb][j][r] = sum of (high + low) over sub-block j.
__device__ __forceinline__ int act_perm(int kl) {
  const int i = kl & 31;
  const int ks_in = i >> 4, rr = i & 15;
  const int c = (rr & 7) >> 1, half = rr >> 3, e = rr & 1;
  return (kl & ~31) + c * 8 + ks_in * 4 + half * 2 + e;
}

__device__ void gemm_prologue(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g, int sb0,
                              int nsb_s, const Smem& sm) {
  const int R = sd.R;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = sb0 * 256, ks = nsb_s * 256;
  const int cstride = act_col_stride(nsb_s);
  __half* act = reinterpret_cast<__half*>(sm.act());
  float* sx = reinterpret_cast<float*>(sm.act() + 2 * R * cstride);
  float* misc = sm.misc();
  if (g.pro == PRO_RMS_X) {
    for (int r = warp; r < R; r += kWarps) {
      const float* x = md.x + static_cast<size_t>(r) * md.H;
      float ss = 0.f;
      for (int k = lane; k < md.H; k += 32) {
        const float v = __ldcg(x + k);
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) misc[r] = 1.0f / sqrtf(ss / static_cast<float>(md.H) + md.eps);
    }
  } else if (g.pro == PRO_GDN_OUT) {
    const int h0 = k0 / md.dv, nh = ks / md.dv;
    for (int p = warp; p < R * nh; p += kWarps) {
      const int r = p / nh, hh = h0 + p % nh;
      const float* o = md.o + static_cast<size_t>(r) * md.o_stride + hh * md.dv;
      float ss = 0.f;
      for (int i = lane; i < md.dv; i += 32) {
        const float v = __ldcg(o + i);
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) misc[p] = 1.0f / sqrtf(ss / static_cast<float>(md.dv) + md.eps);
    }
  }
  __syncthreads();
  const int total = R * ks;
  const int h0 = k0 / (md.dv > 0 ? md.dv : 1), nh = ks / (md.dv > 0 ? md.dv : 1);
  for (int idx = tid; idx < total; idx += kThreads) {
    const int r = idx / ks, kl = idx - r * ks, k = k0 + kl;
    float u;
    if (g.pro == PRO_RMS_X) {
      u = __ldcg(md.x + static_cast<size_t>(r) * md.H + k) * misc[r] * g.gain[k];
    } else if (g.pro == PRO_GDN_OUT) {
      const int hh = k / md.dv, i = k - hh * md.dv;
      const float o = __ldcg(md.o + static_cast<size_t>(r) * md.o_stride + k);
      const float z = __ldcg(md.yin + static_cast<size_t>(r) * md.n_in_max + md.conv_ch + k);
      u = o * misc[r * nh + (hh - h0)] * g.gain[i] * siluf_(z);
    } else if (g.pro == PRO_FA_OUT) {
      const float o = __ldcg(md.o + static_cast<size_t>(r) * md.o_stride + k);
      const float gt = __ldcg(md.yin + static_cast<size_t>(r) * md.n_in_max + md.hq * md.dh + k);
      u = o * sigmoidf_(gt);
    } else {
      u = __ldcg(md.h + static_cast<size_t>(r) * md.F + k);
    }
    const __half hi = __float2half_rn(u);
    const __half lo = __float2half_rn(u - __half2float(hi));
    const int pos = act_perm(kl);
    act[(2 * r) * (cstride / 2) + pos] = hi;
    act[(2 * r + 1) * (cstride / 2) + pos] = lo;
    float s = warp_sum(__half2float(hi) + __half2float(lo));
    if (lane == 0) sx[((kl >> 8) * 8 + ((kl & 255) >> 5)) * R + r] = s;
  }
  __syncthreads();
}

// Number of segments (non-empty warp ranges) that touch tile t, over all
// slices: a unit starts a segment when it is the tile's first unit in its
// slice or when it belongs to a different warp than the unit before it.
__device__ int nseg_of_tile(const GemmDesc& g, const Sched& sc, int grid, int64_t t) {
  int n = 0;
  for (int sl = 0; sl < sc.S; ++sl) {
    const int nsb_s = slice_nsb(sc, g.nsb, sl);
    const int64_t Us = static_cast<int64_t>(g.n_tiles) * nsb_s;
    const int64_t Ws = static_cast<int64_t>(slice_cta0(sc, grid, sl + 1) - slice_cta0(sc, grid, sl)) * kWarps;
    int64_t prev = -1;
    for (int64_t u = t * nsb_s; u < (t + 1) * nsb_s; ++u) {
      const int64_t w = warp_of_unit(Us, Ws, u);
      if (w != prev) ++n;
      prev = w;
    }
  }
  return n;
}

// ------------------------------------------------------------- top-2 state
template <int NR>
struct Top2 {
  float b1[NR];
  int i1[NR];
};

// Larger value wins; on an exact tie the lower vocabulary index wins.
__device__ __forceinline__ void top1_merge(float& a1, int& ai, float b1, int bi) {
  if (b1 > a1 || (b1 == a1 && bi < ai)) {
    a1 = b1;
    ai = bi;
  }
}

// --------------------------------------------------------- GEMM epilogue
template <int NT, bool TOP>
__device__ __forceinline__ void gemm_epilogue(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g,
                                              int64_t tile, const float (&v)[4 * NT], int lane,
                                              Top2<4 * NT>& top) {
  const int R = sd.R;
  const int64_t n = tile * kTileRows + lane;
  switch (g.epi) {
    case EPI_STORE_YIN:
      if (n < g.n_out) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) md.yin[static_cast<size_t>(r) * md.n_in_max + n] = v[r];
      }
      break;
    case EPI_RESID_X:
      if (n < md.H) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) {
            float* p = md.x + static_cast<size_t>(r) * md.H + n;
            *p = __ldcg(p) + v[r];
          }
      }
      break;
    case EPI_SWIGLU_H: {
      const int pos = lane & 15;
      const int64_t f = (tile * 2 + (lane >> 4)) * 8 + (pos & 7);
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) {
        const float up = __shfl_down_sync(0xffffffffu, v[r], 8);
        if (r < R && pos < 8 && f < md.F) md.h[static_cast<size_t>(r) * md.F + f] = siluf_(v[r]) * up;
      }
      break;
    }
    case EPI_TOP2:
      if (TOP && n < md.V) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) {
            const float x = v[r];
            if (!isfinite(x)) atomicOr(&md.err[1], 1);
            top1_merge(top.b1[r], top.i1[r], x, static_cast<int>(n));
            if (md.dbg_logits) md.dbg_logits[static_cast<size_t>(r) * md.V + n] = x;
          }
      }
      break;
  }
}

// ------------------------------------------------------------- GEMM phase
template <int NT>
__device__ void dequant_word(uint32_t w, const uint4& t, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = hfma2_u32(lop3_and_or(w, 0x000F000Fu, 0x64006400u), t.x, t.y);
  a[1] = hfma2_u32(lop3_and_or(w, 0x00F000F0u, 0x64006400u), t.z, t.w);
  a[2] = hfma2_u32(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), t.x, t.y);
  a[3] = hfma2_u32(lop3_and_or(w8, 0x00F000F0u, 0x64006400u), t.z, t.w);
}

template <int NT, bool TOP>
__device__ __forceinline__ bool gemm_phase(const ModelDesc& md, const StepDesc& sd, int gp, const Smem& sm,
                                           WarpCtx& wc) {
  const GemmDesc& g = gemm_desc(md, gp);
  const int R = sd.R;
  const int grid = gridDim.x;
  const Assign a = assign_for(g, R, grid, blockIdx.x, wc.warp);
  produce(wc, md, sd, sm);
  gemm_prologue(md, sd, g, a.sb0, a.nsb_s, sm);

  const int lane = wc.lane, gq = lane >> 2, cq = lane & 3;
  const int cstride = act_col_stride(a.nsb_s);
  const uint8_t* act = sm.act();
  const float* sx = reinterpret_cast<const float*>(act + 2 * R * cstride);
  uint32_t* stab = sm.stab(wc.warp);
  float* dtab = sm.dtab(wc.warp);
  const int orb = lane >> 4, opos = lane & 15, og = opos & 7, ohi = opos >> 3;

  Top2<4 * NT> top;
  if (TOP) {
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) { top.b1[r] = -FLT_MAX; top.i1[r] = 0x7fffffff; }
  }

  float acc[2][NT][4];
  float mn[4 * NT];
  int64_t seg_tile = -1, seg_u0 = 0;

  auto flush = [&](int64_t tile, int64_t u_end) {
    float* stage = reinterpret_cast<float*>(stab);  // [32 rows][16 r]
    __syncwarp();
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r = nt * 4 + cq;
        if (r < R) {
          stage[(rb * 16 + gq) * 16 + r] = acc[rb][nt][0] + acc[rb][nt][1];
          stage[(rb * 16 + gq + 8) * 16 + r] = acc[rb][nt][2] + acc[rb][nt][3];
        }
      }
    __syncwarp();
    float v[4 * NT];
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) v[r] = r < R ? stage[lane * 16 + r] - mn[r] : 0.f;
    __syncwarp();
    const int64_t tu0 = tile * a.nsb_s, tu1 = tu0 + a.nsb_s;
    const bool complete = a.sc.S == 1 && seg_u0 == tu0 && u_end == tu1;
    if (!complete) {
      const int seg_idx = static_cast<int>(tile - a.u0 / a.nsb_s);
      float* slot = md.partial + (static_cast<size_t>(wc.gid) * md.max_seg + seg_idx) * kMaxRows * 32;
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r)
        if (r < R) __stcg(slot + r * 32 + lane, v[r]);
      __threadfence();
      __syncwarp();
      uint32_t last = 0;
      if (lane == 0) {
        const uint32_t n = static_cast<uint32_t>(nseg_of_tile(g, a.sc, grid, tile));
        const uint32_t old = atomicAdd(&md.tickets[tile], 1u);
        last = (old + 1u == n) ? 1u : 0u;
        if (last) md.tickets[tile] = 0u;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) return;
      __threadfence();
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) v[r] = 0.f;
      for (int sl = 0; sl < a.sc.S; ++sl) {
        const int nsb_s = slice_nsb(a.sc, g.nsb, sl);
        const int c0 = slice_cta0(a.sc, grid, sl);
        const int64_t Us = static_cast<int64_t>(g.n_tiles) * nsb_s;
        const int64_t Ws = static_cast<int64_t>(slice_cta0(a.sc, grid, sl + 1) - c0) * kWarps;
        int64_t prev = -1;
        for (int64_t uu = tile * nsb_s; uu < (tile + 1) * nsb_s; ++uu) {
          const int64_t ws = warp_of_unit(Us, Ws, uu);
          if (ws == prev) continue;
          prev = ws;
          const int gid2 = (c0 + static_cast<int>(ws / kWarps)) * kWarps + static_cast<int>(ws % kWarps);
          const int seg2 = static_cast<int>(tile - warp_u0(Us, Ws, ws) / nsb_s);
          const float* s2 = md.partial + (static_cast<size_t>(gid2) * md.max_seg + seg2) * kMaxRows * 32;
#pragma unroll
          for (int r = 0; r < 4 * NT; ++r)
            if (r < R) v[r] += __ldcg(s2 + r * 32 + lane);
        }
      }
    }
    gemm_epilogue<NT, TOP>(md, sd, g, tile, v, lane, top);
  };

  bool ok = true;
  for (int64_t u = a.u0; u < a.u1; ++u) {
    const int64_t tile = u / a.nsb_s;
    const int sbl = static_cast<int>(u - tile * a.nsb_s);
    if (tile != seg_tile) {
      if (seg_tile >= 0) flush(seg_tile, u);
      seg_tile = tile;
      seg_u0 = u;
#pragma unroll
      for (int rb = 0; rb < 2; ++rb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[rb][nt][e] = 0.f;
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) mn[r] = 0.f;
    }
    if (!wait_unit(wc, sm, md, sd.barrier_timeout_ns)) { ok = false; break; }
    const uint8_t* unit = sm.ring(wc.warp, wc.c_pos % kRing);
    // --- own row: scale table, d table and the min term
    {
      const uint4 hdr = *reinterpret_cast<const uint4*>(unit + 16 * lane);
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
      const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
      const uint64_t lo64 = hdr.y | (static_cast<uint64_t>(hdr.z) << 32);
      const uint64_t mid64 = hdr.z | (static_cast<uint64_t>(hdr.w) << 32);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float scf = static_cast<float>(static_cast<uint32_t>(lo64 >> (6 * j)) & 63u);
        const float mf = static_cast<float>(static_cast<uint32_t>(mid64 >> (16 + 6 * j)) & 63u);
        __half2 s2, b2;
        if (ohi == 0) {
          s2 = __float2half2_rn(scf);
          b2 = __float2half2_rn(-1024.f * scf);
        } else {
          s2 = __float2half2_rn(scf * 0.0625f);
          b2 = __float2half2_rn(-64.f * scf);
        }
        uint32_t* e = stab + ((j * 8 + og) * 2 + orb) * 4 + 2 * ohi;
        e[0] = h2u(s2);
        e[1] = h2u(b2);
        const float dm = dmin * mf;  // exact: 11-bit x 6-bit
        const float* sxj = sx + (sbl * 8 + j) * R;
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) mn[r] = fmaf(dm, sxj[r], mn[r]);
      }
      dtab[og * 4 + orb * 2 + ohi] = d;
    }
    __syncwarp();
    float tmp[2][NT][4];
#pragma unroll
    for (int rb = 0; rb < 2; ++rb)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) tmp[rb][nt][e] = 0.f;
    const uint8_t* codes = unit + kUnitHdr;
#pragma unroll (NT <= 2 ? 2 : 1)
    for (int kp = 0; kp < 8; ++kp) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(codes + kp * 512 + lane * 16);
      const uint4 t0 = *reinterpret_cast<const uint4*>(stab + ((kp * 8 + gq) * 2 + 0) * 4);
      const uint4 t1 = *reinterpret_cast<const uint4*>(stab + ((kp * 8 + gq) * 2 + 1) * 4);
      uint4 bf[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int col = nt * 8 + gq;
        if (col < 2 * R)
          bf[nt] = *reinterpret_cast<const uint4*>(act + col * cstride + (sbl * 256 + kp * 32) * 2 + cq * 16);
        else
          bf[nt] = make_uint4(0u, 0u, 0u, 0u);
      }
      uint32_t av[4];
      dequant_word<NT>(w4.x, t0, av);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(tmp[0][nt], av[0], av[1], av[2], av[3], bf[nt].x, bf[nt].y);
      dequant_word<NT>(w4.y, t1, av);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(tmp[1][nt], av[0], av[1], av[2], av[3], bf[nt].x, bf[nt].y);
      dequant_word<NT>(w4.z, t0, av);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(tmp[0][nt], av[0], av[1], av[2], av[3], bf[nt].z, bf[nt].w);
      dequant_word<NT>(w4.w, t1, av);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816(tmp[1][nt], av[0], av[1], av[2], av[3], bf[nt].z, bf[nt].w);
    }
    const float4 d4 = *reinterpret_cast<const float4*>(dtab + gq * 4);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc[0][nt][0] = fmaf(d4.x, tmp[0][nt][0], acc[0][nt][0]);
      acc[0][nt][1] = fmaf(d4.x, tmp[0][nt][1], acc[0][nt][1]);
      acc[0][nt][2] = fmaf(d4.y, tmp[0][nt][2], acc[0][nt][2]);
      acc[0][nt][3] = fmaf(d4.y, tmp[0][nt][3], acc[0][nt][3]);
      acc[1][nt][0] = fmaf(d4.z, tmp[1][nt][0], acc[1][nt][0]);
      acc[1][nt][1] = fmaf(d4.z, tmp[1][nt][1], acc[1][nt][1]);
      acc[1][nt][2] = fmaf(d4.w, tmp[1][nt][2], acc[1][nt][2]);
      acc[1][nt][3] = fmaf(d4.w, tmp[1][nt][3], acc[1][nt][3]);
    }
    __syncwarp();
    ++wc.c_pos;
    produce(wc, md, sd, sm);
  }
  if (ok && seg_tile >= 0) flush(seg_tile, a.u1);

  if (TOP) {
    // warp-level merge, then one record per warp
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) {
      float b1 = top.b1[r];
      int i1 = top.i1[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const int oi1 = __shfl_xor_sync(0xffffffffu, i1, o);
        top1_merge(b1, i1, ob1, oi1);
      }
      if (lane == 0 && r < R) {
        md.top_val[static_cast<size_t>(wc.gid) * kMaxRows + r] = b1;
        md.top_idx[static_cast<size_t>(wc.gid) * kMaxRows + r] = i1;
      }
    }
  }
  return ok;
}

__device__ __forceinline__ bool gemm_dispatch(const ModelDesc& md, const StepDesc& sd, int gp, const Smem& sm,
                                           WarpCtx& wc) {
  const bool top = (gp >> 2) >= md.n_layers;
  switch (sd.nt) {
    case 1: return top ? gemm_phase<1, true>(md, sd, gp, sm, wc) : gemm_phase<1, false>(md, sd, gp, sm, wc);
    case 2: return top ? gemm_phase<2, true>(md, sd, gp, sm, wc) : gemm_phase<2, false>(md, sd, gp, sm, wc);
    default: return top ? gemm_phase<3, true>(md, sd, gp, sm, wc) : gemm_phase<3, false>(md, sd, gp, sm, wc);
  }
}

// ------------------------------------------------------ Gated DeltaNet step
// Per task (sequence, v-head h, 8 rows of the state): causal conv + SiLU of the
// head's q, k (and of the 8 v channels), L2 norms, alpha/beta sigmoids, then
// for each state row the delta rule over the sequence's rows in order:
//   S_i <- alpha S_i + beta (v_i - alpha S_i.k) k,   o_i = S_i.q,
// writing the state after each row into that row's snapshot slot (the commit
// later selects one). Rows of S are independent, so tasks never communicate.
__device__ void gdn_phase(const ModelDesc& md, const StepDesc& sd, int layer, const WarpCtx& wc, const Smem& sm) {
  const LayerDesc& L = md.layer[layer];
  const int gi = L.gdn_i;
  const int hk = md.hk, hv = md.hv, dk = md.dk, dv = md.dv, C = md.conv_ch;
  const int chunks = dv / 8;
  const int per_seq = hv * chunks;
  const int total = sd.n_seq * per_seq;
  const int lane = wc.lane;
  const int ne = dk / 32;  // dims per lane
  const int a_off = C + hv * dv, b_off = a_off + hv;
  const float* cw = L.conv_w;
  for (int task = wc.gid; task < total; task += gridDim.x * kWarps) {
    const int si = task / per_seq, rem = task % per_seq;
    const int h = rem / chunks, i0 = (rem % chunks) * 8;
    const int seq = sd.seq_id[si], T = sd.seq_T[si], row0 = sd.seq_row0[si];
    const int g = h / (hv / hk);
    const size_t seq_slot_in = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_in[si];
    const float* hist = md.conv_state + (seq_slot_in * md.n_gdn + gi) * 3 * C;
    auto pre = [&](int ch, int tau) -> float {
      return tau < 0 ? __ldcg(hist + (3 + tau) * C + ch)
                     : __ldcg(md.yin + static_cast<size_t>(row0 + tau) * md.n_in_max + ch);
    };
    auto conv = [&](int ch, int t) -> float {
      const float* w = cw + ch * 4;
      float c = w[0] * pre(ch, t - 3);
      c = fmaf(w[1], pre(ch, t - 2), c);
      c = fmaf(w[2], pre(ch, t - 1), c);
      c = fmaf(w[3], pre(ch, t), c);
      return siluf_(c);
    };
    // normalised q, k of this head for every row: [t][dk] each, per warp
    float* qs = reinterpret_cast<float*>(sm.phase()) + wc.warp * (2 * kMaxT * 128);
    float* ks = qs + kMaxT * 128;
    float vv[kMaxT], al[kMaxT], be[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (t < T) {
        float q4[4], k4[4];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          q4[e] = k4[e] = 0.f;
          if (e < ne) {
            const int d = lane + 32 * e;
            q4[e] = conv(g * dk + d, t);
            k4[e] = conv(hk * dk + g * dk + d, t);
            sq = fmaf(q4[e], q4[e], sq);
            sk = fmaf(k4[e], k4[e], sk);
          }
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float iq = 1.0f / sqrtf(sq + md.eps), ik = 1.0f / sqrtf(sk + md.eps);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (e < ne) {
            qs[t * 128 + lane + 32 * e] = q4[e] * iq;
            ks[t * 128 + lane + 32 * e] = k4[e] * ik;
          }
        vv[t] = lane < 8 ? conv(2 * hk * dk + h * dv + i0 + lane, t) : 0.f;
        const float* yr = md.yin + static_cast<size_t>(row0 + t) * md.n_in_max;
        al[t] = sigmoidf_(__ldcg(yr + a_off + h));
        be[t] = sigmoidf_(__ldcg(yr + b_off + h));
      }
    }
    __syncwarp();
    const float* Sin = md.gdn_state + ((seq_slot_in * md.n_gdn + gi) * hv + h) * static_cast<size_t>(dv) * dk;
    for (int ii = 0; ii < 8; ++ii) {
      const int i = i0 + ii;
      float s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] = e < ne ? __ldcg(Sin + static_cast<size_t>(i) * dk + lane + 32 * e) : 0.f;
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < T) {
          float kt[4], qt[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            kt[e] = e < ne ? ks[t * 128 + lane + 32 * e] : 0.f;
            qt[e] = e < ne ? qs[t * 128 + lane + 32 * e] : 0.f;
          }
          float sk = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) sk = fmaf(s[e], kt[e], sk);
          sk = warp_sum(sk);
          const float vi = __shfl_sync(0xffffffffu, vv[t], ii);
          const float delta = be[t] * (vi - al[t] * sk);
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e] = fmaf(al[t], s[e], delta * kt[e]);
          float so = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) so = fmaf(s[e], qt[e], so);
          so = warp_sum(so);
          if (lane == 0) md.o[static_cast<size_t>(row0 + t) * md.o_stride + h * dv + i] = so;
          if (sd.seq_snap_all[si] || t == T - 1) {
            const size_t ss = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_out[si][t];
            float* So = md.gdn_state + ((ss * md.n_gdn + gi) * hv + h) * static_cast<size_t>(dv) * dk +
                        static_cast<size_t>(i) * dk;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (e < ne) __stcg(So + lane + 32 * e, s[e]);
          }
        }
      }
    }
    // convolution history after each row, for the channels this task owns
    if (lane < 8) {
      int chs[3];
      int nch = 0;
      chs[nch++] = 2 * hk * dk + h * dv + i0 + lane;
      if (h % (hv / hk) == 0) {
        chs[nch++] = g * dk + i0 + lane;
        chs[nch++] = hk * dk + g * dk + i0 + lane;
      }
      for (int t = 0; t < T; ++t) {
        if (!(sd.seq_snap_all[si] || t == T - 1)) continue;
        const size_t ss = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_out[si][t];
        float* ho = md.conv_state + (ss * md.n_gdn + gi) * 3 * C;
        for (int c = 0; c < nch; ++c)
          for (int j = 0; j < 3; ++j) __stcg(ho + j * C + chs[c], pre(chs[c], t - 2 + j));
      }
    }
    __syncwarp();
  }
}

// -------------------------------------------------------------- attention
// Split-K flash decoding over the paged pool for one (sequence, kv head,
// split): all T x (hq/hkv) query rows of the kv head share every K/V tile of
// 32 tokens; scores and P V run on mma.sync (fp16 in, fp32 accumulate); the
// last split also RoPEs, rounds or quantises and appends this step's own keys
// and values, then attends to them with the causal mask across the draft
// rows. Splits write (m, l, acc) partials; the last block to finish a
// (sequence, head) combines them in split order.
struct AttnSmem {
  __half* Q;   // [48][dh+8]
  __half* K;   // [32][dh+8]
  __half* V;   // [32][dh+8]
  float* S;    // [48][33]
  __half* P;   // [48][40]
  float* m;    // [48]
  float* l;    // [48]
  float* sc;   // [48]
  int* flag;
};

__device__ void attn_store_kv(const ModelDesc& md, int fa_i, int page, int kh, int slot, const float* x,
                              int which, __half* tile_row, int lane) {
  // one warp, dh values in x (global scratch), writes the pool and the f16 tile row
  const int dh = md.dh;
  const size_t row = ((static_cast<size_t>(fa_i) * md.n_pages + page) * md.hkv + kh) * md.page_tokens + slot;
  if (!md.kv_q8) {
    __half* dst = reinterpret_cast<__half*>(which ? md.kv_v : md.kv_k) + row * dh;
    for (int d = lane; d < dh; d += 32) {
      const __half hv = __float2half_rn(x[d]);
      dst[d] = hv;
      tile_row[d] = hv;
    }
  } else {
    int8_t* codes = reinterpret_cast<int8_t*>(which ? md.kv_v : md.kv_k) + row * dh;
    uint16_t* scales = (which ? md.kv_vs : md.kv_ks) + row * (dh / 32);
    for (int b = 0; b < dh / 32; ++b) {
      const float val = x[32 * b + lane];
      const float amax = warp_max(fabsf(val));
      const __half d16 = __double2half(static_cast<double>(amax) / 127.0);
      const double dd = static_cast<double>(__half2float(d16));
      int q = 0;
      if (dd != 0.0) {
        double qq = rint(static_cast<double>(val) / dd);
        qq = qq < -127.0 ? -127.0 : (qq > 127.0 ? 127.0 : qq);
        q = static_cast<int>(qq);
      }
      codes[32 * b + lane] = static_cast<int8_t>(q);
      if (lane == 0) scales[b] = __half_as_ushort(d16);
      tile_row[32 * b + lane] = __float2half_rn(__half2float(d16) * static_cast<float>(q));
    }
  }
}

__device__ void attn_phase(const ModelDesc& md, const StepDesc& sd, int layer, const Smem& sm, float* scratch_row) {
  const LayerDesc& L = md.layer[layer];
  const int fa_i = L.fa_i;
  const int dh = md.dh, hkv = md.hkv, grp = md.hq / md.hkv;
  const int dpad = dh + 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  uint8_t* base = sm.phase();
  AttnSmem as;
  as.Q = reinterpret_cast<__half*>(base);
  as.K = as.Q + kMaxQRows * dpad;
  as.V = as.K + 32 * dpad;
  as.S = reinterpret_cast<float*>(as.V + 32 * dpad);
  as.P = reinterpret_cast<__half*>(as.S + kMaxQRows * 33);
  as.m = reinterpret_cast<float*>(as.P + kMaxQRows * 40);
  as.l = as.m + kMaxQRows;
  as.sc = as.l + kMaxQRows;
  as.flag = reinterpret_cast<int*>(as.sc + kMaxQRows);
  const float inv_sqrt_dh = 1.0f / sqrtf(static_cast<float>(dh));
  const int kq_off = 2 * md.hq * dh;           // k after q and gate
  const int vq_off = kq_off + hkv * dh;         // v after k

  for (int item = blockIdx.x; item < sd.n_attn_items; item += gridDim.x) {
    int si = 0;
    while (si + 1 < sd.n_seq && item >= sd.seq_item0[si + 1]) ++si;
    const int local = item - sd.seq_item0[si];
    const int nsplit = sd.seq_nsplit[si];
    const int kh = local / nsplit, j = local % nsplit;
    const int seq = sd.seq_id[si], T = sd.seq_T[si], row0 = sd.seq_row0[si], Lc = sd.seq_len[si];
    const int qrows = T * grp, mt = (qrows + 15) / 16;
    const int ntile = (Lc + 31) / 32;
    const int tps = sd.seq_tiles_per_split[si];
    const int tb = j * tps, te = min(ntile, tb + tps);
    const bool last = j == nsplit - 1;
    const int* pt = md.page_table + static_cast<size_t>(seq) * md.max_pages_per_seq;

    // Q: RoPE, 1/sqrt(dh), fp16; padding rows zero
    for (int idx = tid; idx < mt * 16 * (dh / 2); idx += kThreads) {
      const int qr = idx / (dh / 2), i = idx % (dh / 2);
      __half qa = __float2half_rn(0.f), qb = qa;
      if (qr < qrows) {
        const int t = qr / grp, hh = kh * grp + qr % grp, row = row0 + t;
        const float* q = md.yin + static_cast<size_t>(row) * md.n_in_max + hh * dh;
        const float a = __ldcg(q + i), b = __ldcg(q + i + dh / 2);
        const float2 cs = sd.rope[row][i];
        qa = __float2half_rn((a * cs.x - b * cs.y) * inv_sqrt_dh);
        qb = __float2half_rn((a * cs.y + b * cs.x) * inv_sqrt_dh);
      }
      as.Q[qr * dpad + i] = qa;
      as.Q[qr * dpad + i + dh / 2] = qb;
    }
    for (int qr = tid; qr < kMaxQRows; qr += kThreads) {
      as.m[qr] = -INFINITY;
      as.l[qr] = 0.f;
    }
    const int nd = dh / kWarps;     // dims per warp in P V
    const int nn = nd / 8;          // n-tiles per warp
    float acc[3][4][4];
#pragma unroll
    for (int a = 0; a < 3; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
    __syncthreads();

    const int n_iter = (te - tb) + (last ? 1 : 0);
    for (int it = 0; it < n_iter; ++it) {
      const bool newtile = last && it == n_iter - 1;
      const int tile = tb + it;
      // ---- load K/V tile (32 tokens) as fp16
      if (!newtile) {
        const int vec_per_row = dh / 8;  // 16-byte vectors of 8 halves
        for (int idx = tid; idx < 2 * 32 * vec_per_row; idx += kThreads) {
          const int which = idx / (32 * vec_per_row);
          const int rem = idx % (32 * vec_per_row);
          const int tk = rem / vec_per_row, vi = rem % vec_per_row;
          const int tok = tile * 32 + tk;
          __half* dst = (which ? as.V : as.K) + tk * dpad + vi * 8;
          uint4 val = make_uint4(0u, 0u, 0u, 0u);
          if (tok < Lc) {
            const int page = pt[tok / md.page_tokens], slot = tok % md.page_tokens;
            const size_t row = ((static_cast<size_t>(fa_i) * md.n_pages + page) * hkv + kh) * md.page_tokens + slot;
            if (!md.kv_q8) {
              const __half* src = reinterpret_cast<const __half*>(which ? md.kv_v : md.kv_k) + row * dh + vi * 8;
              val = __ldcg(reinterpret_cast<const uint4*>(src));
            } else {
              const int8_t* src = reinterpret_cast<const int8_t*>(which ? md.kv_v : md.kv_k) + row * dh + vi * 8;
              const uint2 c8 = __ldcg(reinterpret_cast<const uint2*>(src));
              const uint16_t sbits = __ldcg((which ? md.kv_vs : md.kv_ks) + row * (dh / 32) + (vi * 8) / 32);
              const float d16 = __half2float(__ushort_as_half(sbits));
              __half hv[8];
              const int8_t* cb = reinterpret_cast<const int8_t*>(&c8);
#pragma unroll
              for (int e = 0; e < 8; ++e) hv[e] = __float2half_rn(d16 * static_cast<float>(cb[e]));
              val = *reinterpret_cast<uint4*>(hv);
            }
          }
          *reinterpret_cast<uint4*>(dst) = val;
        }
      } else {
        // this step's own keys/values: RoPE k, round or quantise, append, keep as the tile
        for (int idx = tid; idx < 32 * dh; idx += kThreads) {
          const int tk = idx / dh, d = idx % dh;
          if (tk >= T) {
            as.K[tk * dpad + d] = __float2half_rn(0.f);
            as.V[tk * dpad + d] = __float2half_rn(0.f);
          }
        }
        for (int t = warp; t < T; t += kWarps) {
          const int row = row0 + t, pos = Lc + t;
          const int page = pt[pos / md.page_tokens], slot = pos % md.page_tokens;
          const float* kr = md.yin + static_cast<size_t>(row) * md.n_in_max + kq_off + kh * dh;
          const float* vr = md.yin + static_cast<size_t>(row) * md.n_in_max + vq_off + kh * dh;
          float* ks = scratch_row + warp * 2 * kMaxDh;  // per-warp staging in global scratch
          float* vs = ks + kMaxDh;
          for (int i = lane; i < dh / 2; i += 32) {
            const float a = __ldcg(kr + i), b = __ldcg(kr + i + dh / 2);
            const float2 cs = sd.rope[row][i];
            ks[i] = a * cs.x - b * cs.y;
            ks[i + dh / 2] = a * cs.y + b * cs.x;
          }
          for (int d = lane; d < dh; d += 32) vs[d] = __ldcg(vr + d);
          __syncwarp();
          attn_store_kv(md, fa_i, page, kh, slot, ks, 0, as.K + t * dpad, lane);
          attn_store_kv(md, fa_i, page, kh, slot, vs, 1, as.V + t * dpad, lane);
          __syncwarp();
        }
      }
      __syncthreads();
      // ---- S = Q K^T (scaled already)
      for (int unit = warp; unit < mt * 4; unit += kWarps) {
        const int mi = unit / 4, ni = unit % 4;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k16 = 0; k16 < dh / 16; ++k16) {
          uint32_t a0, a1, a2, a3, b0, b1;
          const int ar = mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ac = k16 * 16 + (lane >> 4) * 8;
          ldsm_x4(a0, a1, a2, a3, as.Q + ar * dpad + ac);
          const int br = ni * 8 + (lane & 7);
          const int bc = k16 * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x2(b0, b1, as.K + br * dpad + bc);
          mma16816(s4, a0, a1, a2, a3, b0, b1);
        }
        const int r0 = mi * 16 + gq, c0 = ni * 8 + 2 * cq;
        as.S[r0 * 33 + c0] = s4[0];
        as.S[r0 * 33 + c0 + 1] = s4[1];
        as.S[(r0 + 8) * 33 + c0] = s4[2];
        as.S[(r0 + 8) * 33 + c0 + 1] = s4[3];
      }
      __syncthreads();
      // ---- online softmax, one row per warp iteration, lane = token
      for (int qr = warp; qr < mt * 16; qr += kWarps) {
        float p = 0.f, scl = 1.f;
        if (qr < qrows) {
          const int t = qr / grp;
          bool valid;
          if (!newtile) valid = tile * 32 + lane < Lc;
          else valid = lane <= t;
          const float s = valid ? as.S[qr * 33 + lane] : -INFINITY;
          const float mx = warp_max(s);
          const float m_old = as.m[qr];
          const float m_new = fmaxf(m_old, mx);
          if (m_new == -INFINITY) {
            p = 0.f;
            scl = 1.f;
          } else {
            p = valid ? expf(s - m_new) : 0.f;
            scl = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
          }
          const float sum = warp_sum(p);
          if (lane == 0) {
            as.l[qr] = as.l[qr] * scl + sum;
            as.m[qr] = m_new;
          }
        }
        as.P[qr * 40 + lane] = __float2half_rn(p);
        if (lane == 0) as.sc[qr] = scl;
      }
      __syncthreads();
      // ---- acc = acc * scale + P V  (warp w owns dims [w*nd, (w+1)*nd))
#pragma unroll
      for (int mi = 0; mi < 3; ++mi) {
        if (mi < mt) {
          const float s0 = as.sc[mi * 16 + gq], s1 = as.sc[mi * 16 + gq + 8];
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) {
            if (ni < nn) {
              acc[mi][ni][0] *= s0;
              acc[mi][ni][1] *= s0;
              acc[mi][ni][2] *= s1;
              acc[mi][ni][3] *= s1;
            }
          }
#pragma unroll
          for (int k16 = 0; k16 < 2; ++k16) {
            uint32_t a0, a1, a2, a3;
            const int ar = mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ac = k16 * 16 + (lane >> 4) * 8;
            ldsm_x4(a0, a1, a2, a3, as.P + ar * 40 + ac);
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
              if (ni < nn) {
                uint32_t b0, b1;
                const int vr = k16 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int vc = warp * nd + ni * 8;
                ldsm_x2_trans(b0, b1, as.V + vr * dpad + vc);
                mma16816(acc[mi][ni], a0, a1, a2, a3, b0, b1);
              }
            }
          }
        }
      }
      __syncthreads();
    }

    // ---- write out: directly if one split, else partial + last-block combine
    if (nsplit == 1) {
#pragma unroll
      for (int mi = 0; mi < 3; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
          if (mi < mt && ni < nn) {
#pragma unroll
            for (int hrow = 0; hrow < 2; ++hrow) {
              const int qr = mi * 16 + gq + hrow * 8;
              if (qr < qrows) {
                const int t = qr / grp, hh = kh * grp + qr % grp;
                const float inv = 1.0f / as.l[qr];
                float* o = md.o + static_cast<size_t>(row0 + t) * md.o_stride + hh * dh + warp * nd + ni * 8 + 2 * cq;
                o[0] = acc[mi][ni][hrow * 2 + 0] * inv;
                o[1] = acc[mi][ni][hrow * 2 + 1] * inv;
              }
            }
          }
    } else {
      float* part = md.attn_part + static_cast<size_t>(item) * kMaxQRows * (kMaxDh + 2);
#pragma unroll
      for (int mi = 0; mi < 3; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
          if (mi < mt && ni < nn) {
#pragma unroll
            for (int hrow = 0; hrow < 2; ++hrow) {
              const int qr = mi * 16 + gq + hrow * 8;
              if (qr < qrows) {
                float* p = part + qr * (kMaxDh + 2) + warp * nd + ni * 8 + 2 * cq;
                __stcg(p, acc[mi][ni][hrow * 2 + 0]);
                __stcg(p + 1, acc[mi][ni][hrow * 2 + 1]);
              }
            }
          }
      for (int qr = tid; qr < qrows; qr += kThreads) {
        __stcg(part + qr * (kMaxDh + 2) + kMaxDh, as.m[qr]);
        __stcg(part + qr * (kMaxDh + 2) + kMaxDh + 1, as.l[qr]);
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int key = si * hkv + kh;
        const uint32_t old = atomicAdd(&md.attn_tickets[key], 1u);
        const int is_last = old + 1u == static_cast<uint32_t>(nsplit);
        if (is_last) md.attn_tickets[key] = 0u;
        *as.flag = is_last;
      }
      __syncthreads();
      if (*as.flag) {
        __threadfence();
        const int item0 = sd.seq_item0[si] + kh * nsplit;
        for (int idx = tid; idx < qrows * dh; idx += kThreads) {
          const int qr = idx / dh, d = idx % dh;
          float M = -INFINITY;
          for (int s = 0; s < nsplit; ++s)
            M = fmaxf(M, __ldcg(md.attn_part + (static_cast<size_t>(item0 + s) * kMaxQRows + qr) * (kMaxDh + 2) + kMaxDh));
          float Ls = 0.f, val = 0.f;
          for (int s = 0; s < nsplit; ++s) {
            const float* p = md.attn_part + (static_cast<size_t>(item0 + s) * kMaxQRows + qr) * (kMaxDh + 2);
            const float ms = __ldcg(p + kMaxDh);
            const float w = ms == -INFINITY ? 0.f : expf(ms - M);
            Ls = fmaf(__ldcg(p + kMaxDh + 1), w, Ls);
            val = fmaf(__ldcg(p + d), w, val);
          }
          const int t = qr / grp, hh = kh * grp + qr % grp;
          md.o[static_cast<size_t>(row0 + t) * md.o_stride + hh * dh + d] = val / Ls;
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ verify
// Block 0: argmax of every row over all warps' top-2 records (lowest index on
// exact ties), then per sequence the longest prefix of drafts that equal the
// previous row's argmax; emitted = accepted drafts + the bonus argmax.
__device__ void verify_phase(const ModelDesc& md, const StepDesc& sd, const Smem& sm) {
  if (blockIdx.x != 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* am = reinterpret_cast<int*>(sm.misc());
  const int nrec = gridDim.x * kWarps;
  for (int r = warp; r < sd.R; r += kWarps) {
    float b1 = -FLT_MAX;
    int i1 = 0x7fffffff;
    for (int gidx = lane; gidx < nrec; gidx += 32) {
      const float v1 = __ldcg(md.top_val + static_cast<size_t>(gidx) * kMaxRows + r);
      const int ix = __ldcg(md.top_idx + static_cast<size_t>(gidx) * kMaxRows + r);
      top1_merge(b1, i1, v1, ix);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob1 = __shfl_xor_sync(0xffffffffu, b1, o);
      const int oi1 = __shfl_xor_sync(0xffffffffu, i1, o);
      top1_merge(b1, i1, ob1, oi1);
    }
    if (lane == 0) am[r] = i1;
  }
  __syncthreads();
  if (tid == 0) {
    int at = 0;
    for (int si = 0; si < sd.n_seq; ++si) {
      const int T = sd.seq_T[si], row0 = sd.seq_row0[si];
      int a = 0;
      while (a + 1 < T && sd.row_tok[row0 + a + 1] == am[row0 + a]) ++a;
      for (int i = 1; i <= a; ++i) md.out[kOutTokens + at++] = sd.row_tok[row0 + i];
      md.out[kOutTokens + at++] = am[row0 + a];
      md.out[kOutCounts + si] = a + 1;
    }
    for (int r = 0; r < sd.R; ++r) md.out[kOutArgmax + r] = am[r];
  }
  if (md.dbg_hidden) {
    for (int idx = tid; idx < sd.R * md.H; idx += kThreads) md.dbg_hidden[idx] = __ldcg(md.x + idx);
  }
}

// ------------------------------------------------------------- the kernel
__global__ void __launch_bounds__(kThreads, 1)
    mk_persistent(const ModelDesc* __restrict__ mdp, const StepDesc* __restrict__ sdp, float* attn_scratch) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int sflag;
  const Smem sm{smem_raw};
  const ModelDesc& md = *mdp;
  const StepDesc& sd = *sdp;
  WarpCtx wc;
  wc.warp = threadIdx.x >> 5;
  wc.lane = threadIdx.x & 31;
  wc.gid = blockIdx.x * kWarps + wc.warp;
  wc.c_pos = wc.p_pos = 0;
  wc.p_gp = -1;
  wc.p_done = false;
  wc.p_u = wc.p_u1 = 0;
  wc.p_nsb_s = wc.p_sb0 = wc.p_nsb = 1;
  wc.p_w = nullptr;
  wc.pol = evict_first_policy();
  if (wc.lane == 0)
    for (int s = 0; s < kRing; ++s) mbar_init(sm.bar(wc.warp, s), 1);
  mbar_fence_init();
  __syncthreads();

  int nbar = 0;
  float* my_scratch = attn_scratch + static_cast<size_t>(blockIdx.x) * kWarps * 2 * kMaxDh;
  produce(wc, md, sd, sm);
  // Phases: 0 embed; then per layer l: 1+5l input GEMM, 2+5l mixer,
  // 3+5l o_proj, 4+5l gate/up, 5+5l down; then lm_head; then verify.
  const int n_phases = 1 + 5 * md.n_layers + 2;
  for (int ph = 0; ph < n_phases; ++ph) {
    bool ok = true;
    int gp = -1;
    if (ph == 0) {
      embed_phase(md, sd, wc);
    } else if (ph == n_phases - 1) {
      verify_phase(md, sd, sm);
      break;
    } else if (ph == n_phases - 2) {
      gp = 4 * md.n_layers;
    } else {
      const int l = (ph - 1) / 5, part = (ph - 1) % 5;
      if (part == 1) {
        produce(wc, md, sd, sm);
        if (md.layer[l].kind == MK_LAYER_GDN) gdn_phase(md, sd, l, wc, sm);
        else attn_phase(md, sd, l, sm, my_scratch);
      } else {
        gp = 4 * l + (part == 0 ? 0 : part - 1);
      }
    }
    if (gp >= 0) ok = gemm_dispatch(md, sd, gp, sm, wc);
    // a failed wait inside a phase still meets the barrier, which reports it
    if (!grid_sync(md, sd, nbar, &sflag) || !ok) break;
  }
  drain(wc, sm, md);
}

cudaError_t launch_persistent(const ModelDesc* md, const StepDesc* sd, float* attn_scratch, int grid,
                              cudaStream_t stream) {
  void* args[] = {const_cast<ModelDesc**>(&md), const_cast<StepDesc**>(&sd), &attn_scratch};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(mk_persistent), dim3(grid), dim3(kThreads), args,
                                     kSmemBytes, stream);
}

cudaError_t configure_persistent(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(mk_persistent),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, reinterpret_cast<const void*>(mk_persistent),
                                                       kThreads, kSmemBytes);
}

}  // namespace mk
