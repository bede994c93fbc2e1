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
// a 4-bit code masked into the low mantissa bits of an fp16 is the exact
// subnormal q * 2^-24 (or q * 2^-20 for the nibble 4 bits up), so one AND per
// pair of weights feeds m16n8k16 directly; the activations are split into two
// fp16 parts (high + low) so that the products stay exact to ~2^-22; each
// 32-wide sub-block's two mma sums are scaled in fp32 by d * sc_j * 2^24 (or
// 2^20), and the min term dmin * sum_j m_j * sum(x over sub-block j) is added
// by the lane that owns the weight row. Weights are used exactly as stored.
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
// Barrier among the math warps only (the producer warp never joins it).
__device__ __forceinline__ void math_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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
  __device__ uint64_t* bar(int warp, int slot) const {  // full: the unit has landed
    return reinterpret_cast<uint64_t*>(base + kOffBar) + warp * kRing + slot;
  }
  __device__ uint64_t* empty(int warp, int slot) const {  // the math warp is done with the slot
    return reinterpret_cast<uint64_t*>(base + kOffBar) + kWarps * kRing + warp * kRing + slot;
  }
  __device__ uint32_t* stab(int warp, int buf) const {
    return reinterpret_cast<uint32_t*>(base + kOffTab + (warp * 2 + buf) * kWarpTab);
  }
  __device__ uint8_t* act() const { return base + kOffAct; }
  __device__ float* misc() const { return reinterpret_cast<float*>(base + kOffMisc); }
  __device__ uint8_t* phase() const { return base + kOffPhase; }
};

// -------------------------------------------------------------- grid sync
// A monotonic arrival counter (zeroed before each launch): barrier n is
// complete when the counter reaches (n+1) * gridDim.x. Arrival is a release
// reduction (no round trip); thread 0 of each block polls with acquire loads.
// An error word set by any block makes every waiter leave; a wait that
// outlives the deadline sets it.
__device__ bool grid_sync(const ModelDesc& md, const StepDesc& sd, int& nbar, int* sflag) {
  math_sync();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile int32_t* err = md.err;
    const uint32_t target = static_cast<uint32_t>(nbar + 1) * gridDim.x;
    const bool skip = sd.skip_block == static_cast<int>(blockIdx.x) && sd.skip_barrier == nbar;
    if (!skip) {
      __threadfence();
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(md.bar) : "memory");
    }
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire(md.bar) >= target) break;
      if ((it & 31u) == 31u) {
        if (*err != 0) { ok = 0; break; }
        const uint64_t now = globaltimer();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > sd.barrier_timeout_ns || it > (1u << 30)) {
          atomicCAS(md.err, 0, DEV_BARRIER_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    if (*err != 0) ok = 0;
    *sflag = ok;
  }
  math_sync();
  ++nbar;
  return *sflag != 0;
}

// ------------------------------------------------------------ the stream
// The producer warp feeds every math warp's ring: lane w (< kWarps) walks math
// warp w's unit sequence over all GEMM phases of the step (the schedule is
// static) and issues one bulk copy per unit as soon as the slot it goes to is
// free, so copies run ahead across grid barriers and mixer phases. Math warps
// wait on the slot's "full" barrier and release it through its "empty" one.
struct WarpCtx {
  int warp, lane, gid;
  uint32_t c_pos;  // units consumed by this math warp
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
  uint32_t Us, Ws, ws, u0, u1;
};

__device__ __forceinline__ Assign assign_for(const GemmDesc& g, int R, int grid, int cta, int warp) {
  Assign a;
  a.sc = make_sched(g.nsb, R);
  a.sl = slice_of_cta(a.sc, grid, cta);
  a.cta0 = slice_cta0(a.sc, grid, a.sl);
  const int cta1 = slice_cta0(a.sc, grid, a.sl + 1);
  a.nsb_s = slice_nsb(a.sc, g.nsb, a.sl);
  a.sb0 = slice_sb0(a.sc, a.sl);
  a.Us = static_cast<uint32_t>(g.n_tiles) * a.nsb_s;
  a.Ws = static_cast<uint32_t>(cta1 - a.cta0) * kWarps;
  a.ws = static_cast<uint32_t>(cta - a.cta0) * kWarps + warp;
  a.u0 = warp_u0(a.Us, a.Ws, a.ws);
  a.u1 = warp_u0(a.Us, a.Ws, a.ws + 1);
  return a;
}

// Bounded wait for an mbarrier phase; false (and the error word set) on timeout
// or when another block has already reported an error.
__device__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity, const ModelDesc& md, uint64_t timeout_ns,
                                  int32_t code) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  volatile int32_t* err = md.err;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0 && *err != 0) return false;
    if (globaltimer() - t0 > timeout_ns || it > (1u << 26)) {
      atomicCAS(md.err, 0, code);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Lanes 0..kWarps-1 each walk one math warp's unit sequence; the warp stays
// converged: every sweep, each lane issues its next unit if that unit's slot
// has been released, then the sweep repeats until every lane is done.
__device__ void producer_warp(const ModelDesc& md, const StepDesc& sd, const Smem& sm) {
  const int lane = threadIdx.x & 31;
  const int w = lane < kWarps ? lane : 0;
  const uint64_t pol = evict_first_policy();
  int gp = -1;
  uint32_t left = 0, tile = 0, sbl = 0, p = 0;
  int nsb_s = 1, sb0 = 0, nsb = 1;
  const uint8_t* wsrc = nullptr;
  bool done = lane >= kWarps;
  volatile int32_t* err = md.err;
  uint64_t t_idle = 0;
  for (uint32_t sweep = 0;; ++sweep) {
    // advance to the next phase with units for this lane's warp
    while (!done && left == 0) {
      if (++gp > 4 * md.n_layers) { done = true; break; }
      const GemmDesc& g = gemm_desc(md, gp);
      const Assign a = assign_for(g, sd.R, gridDim.x, blockIdx.x, w);
      left = a.u1 - a.u0;
      nsb_s = a.nsb_s;
      tile = a.u0 / nsb_s;
      sbl = a.u0 - tile * nsb_s;
      sb0 = a.sb0;
      nsb = g.nsb;
      wsrc = g.w;
    }
    if (__all_sync(0xffffffffu, done)) break;
    bool issued = false;
    if (!done) {
      const int slot = p % kRing;
      if (mbar_test(sm.empty(w, slot), ((p / kRing) & 1u) ^ 1u)) {
        uint64_t* b = sm.bar(w, slot);
        mbar_arrive_expect_tx(b, kUnitBytes);
        bulk_g2s(sm.ring(w, slot), wsrc + (static_cast<size_t>(tile) * nsb + sb0 + sbl) * kUnitBytes, kUnitBytes,
                 b, pol);
        if (++sbl == static_cast<uint32_t>(nsb_s)) { sbl = 0; ++tile; }
        --left;
        ++p;
        issued = true;
      }
    }
    if (__any_sync(0xffffffffu, issued)) {
      t_idle = 0;
    } else if ((sweep & 63u) == 63u) {
      // nothing could be issued: the math warps are behind; give up only on
      // an error or after the deadline
      if (*err != 0) break;
      const uint64_t now = globaltimer();
      if (t_idle == 0) t_idle = now;
      else if (now - t_idle > sd.barrier_timeout_ns) { atomicCAS(md.err, 0, DEV_COPY_TIMEOUT); break; }
    }
  }
  // the block must not exit while a copy into its shared memory is in flight
  if (lane < kWarps)
    for (uint32_t q = p > static_cast<uint32_t>(kRing) ? p - kRing : 0; q < p; ++q)
      mbar_wait_bounded(sm.bar(w, q % kRing), (q / kRing) & 1u, md, 50000000ull, DEV_COPY_TIMEOUT);
}

__device__ __forceinline__ bool wait_unit(const WarpCtx& wc, const Smem& sm, const ModelDesc& md,
                                          uint64_t timeout_ns) {
  return mbar_wait_bounded(sm.bar(wc.warp, wc.c_pos % kRing), (wc.c_pos / kRing) & 1u, md, timeout_ns,
                           DEV_COPY_TIMEOUT);
}

// The math warp is done reading its current slot.
__device__ __forceinline__ void release_unit(WarpCtx& wc, const Smem& sm) {
  __syncwarp();
  if (wc.lane == 0) mbar_arrive(sm.empty(wc.warp, wc.c_pos % kRing));
  ++wc.c_pos;
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
    float sq = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = i0 + e;
      const uint8_t byte = __ldg(blk + 16 + 16 * j + (i % 16));
      const int q = i < 16 ? (byte & 15) : (byte >> 4);
      const float xv = ds * static_cast<float>(q) - dm;
      md.x[static_cast<size_t>(r) * md.H + sb * 256 + 32 * j + i] = xv;
      sq = fmaf(xv, xv, sq);
    }
    // the 4 lanes of sub-block j hold one 32-wide chunk
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    if ((wc.lane & 3) == 0) md.xsq[static_cast<size_t>(sb * 8 + j) * kMaxRows + r] = sq;
  }
}

// --------------------------------------------------------- GEMM prologue
// Fills the activation region for reduction slice [sb0, sb0 + nsb_s): for each
// row r, column 2r holds the fp16 high part and column 2r+1 the low part of the
// input vector, each column in the per-32 permuted order of the B fragments;
// then sx[sb][j][r] = sum of (high + low) over sub-block j. Loads are float4,
// and per-row norms reduce over the whole block in a fixed order.
__device__ __forceinline__ int act_perm(int kl) {
  const int i = kl & 31;
  const int ks_in = i >> 4, rr = i & 15;
  const int c = (rr & 7) >> 1, half = rr >> 3, e = rr & 1;
  return (kl & ~31) + c * 8 + ks_in * 4 + half * 2 + e;
}

__device__ __forceinline__ void put_act(__half* act, int cs2, int R, float* sx, int r, int kl, const float (&u)[4],
                                        int lane) {
  __half hi[4], lo[4];
  float part = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi[e] = __float2half_rn(u[e]);
    lo[e] = __float2half_rn(u[e] - __half2float(hi[e]));
    part += __half2float(hi[e]) + __half2float(lo[e]);
  }
  // k and k+1 (and k+2, k+3) are adjacent pairs in the permuted order
  const int p0 = act_perm(kl), p2 = act_perm(kl + 2);
  __half* chi = act + (2 * r) * cs2;
  __half* clo = act + (2 * r + 1) * cs2;
  *reinterpret_cast<__half2*>(chi + p0) = __halves2half2(hi[0], hi[1]);
  *reinterpret_cast<__half2*>(chi + p2) = __halves2half2(hi[2], hi[3]);
  *reinterpret_cast<__half2*>(clo + p0) = __halves2half2(lo[0], lo[1]);
  *reinterpret_cast<__half2*>(clo + p2) = __halves2half2(lo[2], lo[3]);
  // 8 consecutive threads hold one 32-wide sub-block
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  part += __shfl_xor_sync(0xffffffffu, part, 4);
  if ((lane & 7) == 0) sx[((kl >> 8) * 8 + ((kl & 255) >> 5)) * R + r] = part;
}

// One round of loads: every thread issues all of its source float4 loads
// (up to kB groups, plus the per-chunk sums of squares for an RMSNorm) before
// using any of them, so the prologue costs about one L2 round trip.
// RMSNorm: 1/rms from the 32-wide chunk sums the residual writers left, added
// in a fixed order. Gated DeltaNet output: each head's 128 (or 64) values are
// the float4s of 32 (or 16) consecutive lanes, so its norm is a shuffle sum.
__device__ void gemm_prologue(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g, int sb0,
                              int nsb_s, const Smem& sm) {
  constexpr int kB = 8;
  const int R = sd.R;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = sb0 * 256, ks = nsb_s * 256;
  const int cstride = act_col_stride(nsb_s);
  __half* act = reinterpret_cast<__half*>(sm.act());
  float* sx = reinterpret_cast<float*>(sm.act() + 2 * R * cstride);
  float* misc = sm.misc();                        // 1/rms per row
  float* red = misc + 1024 - kWarps * kMaxRows;   // [warp][row] partial sums
  const int per_row = ks / 4;
  const int cs2 = cstride / 2;
  const int total = R * per_row;
  const int nchunk = md.H / 32;
  for (int base = 0; base < total; base += kThreads * kB) {
    float4 s1[kB], s2[kB];
    float sq[kMaxRows];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int idx = base + b * kThreads + tid;
      s1[b] = s2[b] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < total) {
        const int r = idx / per_row, k = k0 + (idx - r * per_row) * 4;
        if (g.pro == PRO_RMS_X) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.x + static_cast<size_t>(r) * md.H + k));
        } else if (g.pro == PRO_GDN_OUT) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.o + static_cast<size_t>(r) * md.o_stride + k));
          s2[b] = __ldcg(reinterpret_cast<const float4*>(md.yin + static_cast<size_t>(r) * md.n_in_max + md.conv_ch + k));
        } else if (g.pro == PRO_FA_OUT) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.o + static_cast<size_t>(r) * md.o_stride + k));
          s2[b] = __ldcg(reinterpret_cast<const float4*>(md.yin + static_cast<size_t>(r) * md.n_in_max + md.hq * md.dh + k));
        } else {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.h + static_cast<size_t>(r) * md.F + k));
        }
      }
    }
    if (g.pro == PRO_RMS_X && base == 0) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        sq[r] = 0.f;
        if (r < R)
          for (int c = tid; c < nchunk; c += kThreads) sq[r] += __ldcg(md.xsq + static_cast<size_t>(c) * kMaxRows + r);
      }
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
        if (r < R) {
          const float t = warp_sum(sq[r]);
          if (lane == 0) red[warp * kMaxRows + r] = t;
        }
      math_sync();
      if (tid < R) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += red[w * kMaxRows + tid];
        misc[tid] = 1.0f / sqrtf(t / static_cast<float>(md.H) + md.eps);
      }
      math_sync();
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int idx = base + b * kThreads + tid;
      if (idx < total) {  // warp-uniform: total is a multiple of 64
        const int r = idx / per_row, kl = (idx - r * per_row) * 4, k = k0 + kl;
        float u[4];
        if (g.pro == PRO_RMS_X) {
          const float4 gg = *reinterpret_cast<const float4*>(g.gain + k);
          const float sc = misc[r];
          u[0] = s1[b].x * sc * gg.x; u[1] = s1[b].y * sc * gg.y; u[2] = s1[b].z * sc * gg.z; u[3] = s1[b].w * sc * gg.w;
        } else if (g.pro == PRO_GDN_OUT) {
          float hs = fmaf(s1[b].x, s1[b].x, fmaf(s1[b].y, s1[b].y, fmaf(s1[b].z, s1[b].z, s1[b].w * s1[b].w)));
          for (int off = 1; off < md.dv / 4; off <<= 1) hs += __shfl_xor_sync(0xffffffffu, hs, off);
          const float sc = 1.0f / sqrtf(hs / static_cast<float>(md.dv) + md.eps);
          const int i = k % md.dv;
          const float4 gg = *reinterpret_cast<const float4*>(g.gain + i);
          u[0] = s1[b].x * sc * gg.x * siluf_(s2[b].x); u[1] = s1[b].y * sc * gg.y * siluf_(s2[b].y);
          u[2] = s1[b].z * sc * gg.z * siluf_(s2[b].z); u[3] = s1[b].w * sc * gg.w * siluf_(s2[b].w);
        } else if (g.pro == PRO_FA_OUT) {
          u[0] = s1[b].x * sigmoidf_(s2[b].x); u[1] = s1[b].y * sigmoidf_(s2[b].y);
          u[2] = s1[b].z * sigmoidf_(s2[b].z); u[3] = s1[b].w * sigmoidf_(s2[b].w);
        } else {
          u[0] = s1[b].x; u[1] = s1[b].y; u[2] = s1[b].z; u[3] = s1[b].w;
        }
        put_act(act, cs2, R, sx, r, kl, u, lane);
      }
    }
  }
  math_sync();
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
                                              uint32_t tile, const float (&v)[4 * NT], int lane,
                                              Top2<4 * NT>& top) {
  const int R = sd.R;
  const int n = static_cast<int>(tile) * kTileRows + lane;
  switch (g.epi) {
    case EPI_STORE_YIN:
      if (n < g.n_out) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) md.yin[static_cast<size_t>(r) * md.n_in_max + n] = v[r];
      }
      break;
    case EPI_RESID_X: {
      // H is a multiple of 256, so every lane of the tile holds a real row
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r)
        if (r < R) {
          float* p = md.x + static_cast<size_t>(r) * md.H + n;
          const float xn = __ldcg(p) + v[r];
          *p = xn;
          const float sq = warp_sum(xn * xn);  // the next RMSNorm's partial for this 32-wide chunk
          if (lane == 0) md.xsq[static_cast<size_t>(tile) * kMaxRows + r] = sq;
        }
      break;
    }
    case EPI_SWIGLU_H: {
      const int pos = lane & 15;
      const int f = (static_cast<int>(tile) * 2 + (lane >> 4)) * 8 + (pos & 7);
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
            top1_merge(top.b1[r], top.i1[r], x, n);
            if (md.dbg_logits) md.dbg_logits[static_cast<size_t>(r) * md.V + n] = x;
          }
      }
      break;
  }
}

// ------------------------------------------------------------- GEMM phase
// One word of 8 codes -> the four A registers of a 16x16 block, exactly: a
// code masked into the low mantissa bits of an fp16 is the subnormal value
// q * 2^-24 (rows g, nibbles at bits 0-3 / 16-19) or q * 2^-20 (rows g+8,
// nibbles at bits 4-7 / 20-23); the tensor core multiplies subnormals
// exactly, and the per-row factor 2^24 or 2^20 goes into the fp32 scale.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = w & 0x000F000Fu;
  a[1] = w & 0x00F000F0u;
  a[2] = w8 & 0x000F000Fu;
  a[3] = w8 & 0x00F000F0u;
}


// One step of the own-row header decode: sub-block j of the lane's row in
// the next unit -> its fp32 scale d * sc_j * 2^24 (or 2^20), exact, into the
// scale table, and the min term dmin * m_j * sum_j(x) added into mtmp.
template <int NT>
__device__ __forceinline__ float decode_step(int j, const uint4& hdr, float dscale, float dmin, const float* sxb,
                                             int R, float (&mtmp)[4 * NT]) {
  const uint32_t f0 = hdr.y, f1 = hdr.z, f2 = hdr.w;
  uint32_t sc, m;
  switch (j) {  // 6-bit fields: sc_j at bit 6j, m_j at bit 48 + 6j of the 96-bit field
    case 0: sc = f0 & 63u; m = (f1 >> 16) & 63u; break;
    case 1: sc = (f0 >> 6) & 63u; m = (f1 >> 22) & 63u; break;
    case 2: sc = (f0 >> 12) & 63u; m = __funnelshift_r(f1, f2, 28) & 63u; break;
    case 3: sc = (f0 >> 18) & 63u; m = (f2 >> 2) & 63u; break;
    case 4: sc = (f0 >> 24) & 63u; m = (f2 >> 8) & 63u; break;
    case 5: sc = __funnelshift_r(f0, f1, 30) & 63u; m = (f2 >> 14) & 63u; break;
    case 6: sc = (f1 >> 4) & 63u; m = (f2 >> 20) & 63u; break;
    default: sc = (f1 >> 10) & 63u; m = (f2 >> 26) & 63u; break;
  }
  const float dm = dmin * static_cast<float>(m);  // exact: 11-bit x 6-bit
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r)
    if (r < R) mtmp[r] = fmaf(dm, sxb[j * R + r], mtmp[r]);
  return dscale * static_cast<float>(sc);  // exact: 11-bit x 6-bit
}

// The own row's 8 sub-block scales go to the scale table in one burst, after
// the loop that computed them: no shared store sits between the loop's loads.
__device__ __forceinline__ void store_scales(float* tab, const float (&scl)[8], int og, int orb, int ohi) {
#pragma unroll
  for (int j = 0; j < 8; ++j) tab[j * 32 + og * 4 + orb * 2 + ohi] = scl[j];
}

// Out of line: each phase function is entered once per phase, and its own
// register allocation keeps the hot loops free of spills.
//
// Per math warp, software-pipelined over its units: while the mma loop of
// unit k runs, the own-row header decode of unit k+1 fills the other scale
// table, so neither the decode latency nor the tail of the mma chains stalls
// the warp.
template <int NT, bool TOP>
__device__ __noinline__ bool gemm_phase(const ModelDesc& md, const StepDesc& sd, int gp, const Smem& sm,
                                        WarpCtx& wc) {
  const GemmDesc& g = gemm_desc(md, gp);
  const int R = sd.R;
  const int grid = gridDim.x;
  const Assign a = assign_for(g, R, grid, blockIdx.x, wc.warp);
  gemm_prologue(md, sd, g, a.sb0, a.nsb_s, sm);

  const int lane = wc.lane, gq = lane >> 2, cq = lane & 3;
  const int cstride = act_col_stride(a.nsb_s);
  const uint8_t* act = sm.act();
  const float* sx = reinterpret_cast<const float*>(act + 2 * R * cstride);
  // own row of this lane inside a tile: half rb, position og + 8*ohi; its
  // codes enter the mma as q * 2^-24 (ohi = 0) or q * 2^-20 (ohi = 1)
  const int orb = lane >> 4, opos = lane & 15, og = opos & 7, ohi = opos >> 3;
  const float row_unscale = ohi ? 1048576.0f : 16777216.0f;  // 2^20 or 2^24
  const int nsb_s = a.nsb_s;
  // B column of this lane per column tile; columns past 2R read column 2R-1
  // (their products land in output columns nobody reads)
  const uint8_t* bcol[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) bcol[nt] = act + min(nt * 8 + gq, 2 * R - 1) * cstride + cq * 16;

  Top2<4 * NT> top;
  if (TOP) {
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) { top.b1[r] = -FLT_MAX; top.i1[r] = 0x7fffffff; }
  }

  float acc[2][NT][4];
  float mn[4 * NT], mtmp[4 * NT];
  uint32_t seg_u0 = a.u0;
#pragma unroll
  for (int rb = 0; rb < 2; ++rb)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rb][nt][e] = 0.f;

  auto flush = [&](uint32_t tile, uint32_t u_end, float* stage) {
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
    const uint32_t tu0 = tile * nsb_s, tu1 = tu0 + nsb_s;
    const bool complete = a.sc.S == 1 && seg_u0 == tu0 && u_end == tu1;
    if (!complete) {
      const int seg_idx = static_cast<int>(tile - a.u0 / nsb_s);
      float* slot = md.partial + (static_cast<size_t>(wc.gid) * md.max_seg + seg_idx) * kMaxRows * 32;
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r)
        if (r < R) __stcg(slot + r * 32 + lane, v[r]);
      __threadfence();
      __syncwarp();
      uint32_t last = 0;
      if (lane == 0) {
        uint32_t n = 0;
        for (int sl = 0; sl < a.sc.S; ++sl) {
          const uint32_t ns = slice_nsb(a.sc, g.nsb, sl);
          const uint32_t Us = static_cast<uint32_t>(g.n_tiles) * ns;
          const uint32_t Ws =
              static_cast<uint32_t>(slice_cta0(a.sc, grid, sl + 1) - slice_cta0(a.sc, grid, sl)) * kWarps;
          n += segments_in(Us, Ws, tile * ns, tile * ns + ns);
        }
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
        const uint32_t ns = slice_nsb(a.sc, g.nsb, sl);
        const int c0 = slice_cta0(a.sc, grid, sl);
        const uint32_t Us = static_cast<uint32_t>(g.n_tiles) * ns;
        const uint32_t Ws = static_cast<uint32_t>(slice_cta0(a.sc, grid, sl + 1) - c0) * kWarps;
        const uint32_t ua = tile * ns, ub = ua + ns;
        // warps holding units [ua, ub), in order: one per unit when ranges
        // hold at most one unit, else the consecutive run wf..wl
        const bool sparse = Us < Ws;
        const uint32_t first = sparse ? ua : warp_of_unit(Us, Ws, ua);
        const uint32_t last_w = sparse ? ub - 1 : warp_of_unit(Us, Ws, ub - 1);
        for (uint32_t it = first; it <= last_w; ++it) {
          const uint32_t ws = sparse ? warp_of_unit(Us, Ws, it) : it;
          const int gid2 = (c0 + static_cast<int>(ws / kWarps)) * kWarps + static_cast<int>(ws % kWarps);
          const int seg2 = static_cast<int>(tile - warp_u0(Us, Ws, ws) / ns);
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
  if (a.u1 > a.u0) {
    uint32_t tile = a.u0 / nsb_s;
    int sbl = static_cast<int>(a.u0 - tile * nsb_s);
    // pipeline fill: decode the first unit
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) mtmp[r] = 0.f;
    if (!wait_unit(wc, sm, md, sd.barrier_timeout_ns)) {
      ok = false;
    } else {
      const uint8_t* unit = sm.ring(wc.warp, wc.c_pos % kRing);
      const uint4 hdr = *reinterpret_cast<const uint4*>(unit + 16 * lane);
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
      const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
      float scl[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) scl[j] = decode_step<NT>(j, hdr, d * row_unscale, dmin, sx + sbl * 8 * R, R, mtmp);
      store_scales(reinterpret_cast<float*>(sm.stab(wc.warp, 0)), scl, og, orb, ohi);
    }
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) mn[r] = mtmp[r];
    __syncwarp();
    for (uint32_t u = a.u0; ok && u < a.u1; ++u) {
      const int cur = static_cast<int>((u - a.u0) & 1u);
      const bool has_next = u + 1 < a.u1;
      const int sbl_next = sbl + 1 == nsb_s ? 0 : sbl + 1;
      const uint8_t* unit = sm.ring(wc.warp, wc.c_pos % kRing);
      const float* tab = reinterpret_cast<const float*>(sm.stab(wc.warp, cur));
      float* tabn = reinterpret_cast<float*>(sm.stab(wc.warp, cur ^ 1));
      uint4 hdrn = make_uint4(0u, 0u, 0u, 0u);
      float dscalen = 0.f, dminn = 0.f;
      if (has_next) {
        WarpCtx nx = wc;
        ++nx.c_pos;
        if (!wait_unit(nx, sm, md, sd.barrier_timeout_ns)) { ok = false; break; }
        hdrn = *reinterpret_cast<const uint4*>(sm.ring(wc.warp, nx.c_pos % kRing) + 16 * lane);
        dscalen = __half2float(__ushort_as_half(static_cast<unsigned short>(hdrn.x & 0xffffu))) * row_unscale;
        dminn = __half2float(__ushort_as_half(static_cast<unsigned short>(hdrn.x >> 16)));
      }
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) mtmp[r] = 0.f;
      const uint8_t* codes = unit + kUnitHdr + lane * 16;
      const int boff = sbl * 512;
      const float* sxn = sx + sbl_next * 8 * R;
      float scl[8];
#pragma unroll
      for (int kp = 0; kp < 8; ++kp) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(codes + kp * 512);
        // fp32 scales of rows (g, g+8) of both 16-row halves for sub-block kp
        const float4 s4 = *reinterpret_cast<const float4*>(tab + kp * 32 + gq * 4);
        uint4 bf[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          bf[nt] = *reinterpret_cast<const uint4*>(bcol[nt] + boff + kp * 64);
        float t0[NT][4], t1[NT][4];  // sub-block sums of halves 0 and 1 (two k-steps each)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) t0[nt][e] = t1[nt][e] = 0.f;
        uint32_t av[4];
        dequant_word(w4.x, av);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(t0[nt], av[0], av[1], av[2], av[3], bf[nt].x, bf[nt].y);
        dequant_word(w4.y, av);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(t1[nt], av[0], av[1], av[2], av[3], bf[nt].x, bf[nt].y);
        dequant_word(w4.z, av);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(t0[nt], av[0], av[1], av[2], av[3], bf[nt].z, bf[nt].w);
        dequant_word(w4.w, av);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(t1[nt], av[0], av[1], av[2], av[3], bf[nt].z, bf[nt].w);
        scl[kp] = has_next ? decode_step<NT>(kp, hdrn, dscalen, dminn, sxn, R, mtmp) : 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[0][nt][0] = fmaf(s4.x, t0[nt][0], acc[0][nt][0]);
          acc[0][nt][1] = fmaf(s4.x, t0[nt][1], acc[0][nt][1]);
          acc[0][nt][2] = fmaf(s4.y, t0[nt][2], acc[0][nt][2]);
          acc[0][nt][3] = fmaf(s4.y, t0[nt][3], acc[0][nt][3]);
          acc[1][nt][0] = fmaf(s4.z, t1[nt][0], acc[1][nt][0]);
          acc[1][nt][1] = fmaf(s4.z, t1[nt][1], acc[1][nt][1]);
          acc[1][nt][2] = fmaf(s4.w, t1[nt][2], acc[1][nt][2]);
          acc[1][nt][3] = fmaf(s4.w, t1[nt][3], acc[1][nt][3]);
        }
      }
      if (has_next) store_scales(tabn, scl, og, orb, ohi);
      release_unit(wc, sm);  // includes __syncwarp: both tables are settled
      if (++sbl == nsb_s || u + 1 == a.u1) {
        flush(tile, u + 1, reinterpret_cast<float*>(sm.stab(wc.warp, cur)));
        seg_u0 = u + 1;
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[rb][nt][e] = 0.f;
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r) mn[r] = 0.f;
        if (sbl == nsb_s) { sbl = 0; ++tile; }
      }
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) mn[r] += mtmp[r];
      __syncwarp();
    }
  }

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
__device__ __noinline__ void gdn_phase(const ModelDesc& md, const StepDesc& sd, int layer, const WarpCtx& wc, const Smem& sm) {
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
    float* qs = reinterpret_cast<float*>(sm.phase()) + wc.warp * (2 * kMaxT * 128 + kMaxT * 10);
    float* ks = qs + kMaxT * 128;
    // per-row gates and this task's 8 v values: [t] in shared memory after q, k
    float* vs = ks + kMaxT * 128;  // [kMaxT][8]
    float* gs = vs + kMaxT * 8;    // [kMaxT][2] alpha, beta
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
        if (lane < 8) vs[t * 8 + lane] = conv(2 * hk * dk + h * dv + i0 + lane, t);
        if (lane == 0) {
          const float* yr = md.yin + static_cast<size_t>(row0 + t) * md.n_in_max;
          gs[t * 2 + 0] = sigmoidf_(__ldcg(yr + a_off + h));
          gs[t * 2 + 1] = sigmoidf_(__ldcg(yr + b_off + h));
        }
      }
    }
    __syncwarp();
    const float* Sin = md.gdn_state + ((seq_slot_in * md.n_gdn + gi) * hv + h) * static_cast<size_t>(dv) * dk;
    // the task's 8 state rows, loaded at once (independent rows of S)
    float s[8][4];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        s[ii][e] = e < ne ? __ldcg(Sin + static_cast<size_t>(i0 + ii) * dk + lane + 32 * e) : 0.f;
    for (int t = 0; t < T; ++t) {
      float kt[4], qt[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kt[e] = e < ne ? ks[t * 128 + lane + 32 * e] : 0.f;
        qt[e] = e < ne ? qs[t * 128 + lane + 32 * e] : 0.f;
      }
      const float al = gs[t * 2 + 0], be = gs[t * 2 + 1];
      const bool snap = sd.seq_snap_all[si] || t == T - 1;
      float* So = nullptr;
      if (snap) {
        const size_t ss = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_out[si][t];
        So = md.gdn_state + ((ss * md.n_gdn + gi) * hv + h) * static_cast<size_t>(dv) * dk;
      }
      float skv[8];
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) a = fmaf(s[ii][e], kt[e], a);
        skv[ii] = a;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) skv[ii] += __shfl_xor_sync(0xffffffffu, skv[ii], o);
      float sov[8];
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const float delta = be * (vs[t * 8 + ii] - al * skv[ii]);
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s[ii][e] = fmaf(al, s[ii][e], delta * kt[e]);
          a = fmaf(s[ii][e], qt[e], a);
        }
        sov[ii] = a;
        if (snap) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (e < ne) __stcg(So + static_cast<size_t>(i0 + ii) * dk + lane + 32 * e, s[ii][e]);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) sov[ii] += __shfl_xor_sync(0xffffffffu, sov[ii], o);
      if (lane < 8) {
        float ov = sov[0];
#pragma unroll
        for (int ii = 1; ii < 8; ++ii) ov = lane == ii ? sov[ii] : ov;
        md.o[static_cast<size_t>(row0 + t) * md.o_stride + h * dv + i0 + lane] = ov;
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

__device__ __noinline__ void attn_phase(const ModelDesc& md, const StepDesc& sd, int layer, const Smem& sm, float* scratch_row) {
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
  float* wbuf = reinterpret_cast<float*>(as.flag + 4);  // [kWarps][kMaxSplits] split weights
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
    math_sync();

    const int n_iter = (te - tb) + (last ? 1 : 0);
    // K/V tile staging: each thread holds up to 8 raw 16-byte (fp16) or
    // 8-byte (q8, plus its block scale) vectors of the NEXT cached tile in
    // registers, so the tile's load latency overlaps the current tile's work.
    const int vec_per_row = dh / 8;
    const int nvec = 2 * 32 * vec_per_row;  // K and V rows of 32 tokens
    uint4 pf[8];
    uint16_t pfs[8];
    auto load_tile = [&](int tile) {
#pragma unroll
      for (int jv = 0; jv < 8; ++jv) {
        const int idx = tid + jv * kThreads;
        pf[jv] = make_uint4(0u, 0u, 0u, 0u);
        pfs[jv] = 0;
        if (idx < nvec) {
          const int which = idx / (32 * vec_per_row);
          const int rem = idx % (32 * vec_per_row);
          const int tk = rem / vec_per_row, vi = rem % vec_per_row;
          const int tok = tile * 32 + tk;
          if (tok < Lc) {
            const int page = pt[tok / md.page_tokens], slot = tok % md.page_tokens;
            const size_t row = ((static_cast<size_t>(fa_i) * md.n_pages + page) * hkv + kh) * md.page_tokens + slot;
            if (!md.kv_q8) {
              pf[jv] = __ldcg(reinterpret_cast<const uint4*>(
                  reinterpret_cast<const __half*>(which ? md.kv_v : md.kv_k) + row * dh + vi * 8));
            } else {
              const uint2 c8 = __ldcg(reinterpret_cast<const uint2*>(
                  reinterpret_cast<const int8_t*>(which ? md.kv_v : md.kv_k) + row * dh + vi * 8));
              pf[jv].x = c8.x;
              pf[jv].y = c8.y;
              pfs[jv] = __ldcg((which ? md.kv_vs : md.kv_ks) + row * (dh / 32) + (vi * 8) / 32);
            }
          }
        }
      }
    };
    auto store_tile = [&]() {
#pragma unroll
      for (int jv = 0; jv < 8; ++jv) {
        const int idx = tid + jv * kThreads;
        if (idx < nvec) {
          const int which = idx / (32 * vec_per_row);
          const int rem = idx % (32 * vec_per_row);
          const int tk = rem / vec_per_row, vi = rem % vec_per_row;
          __half* dst = (which ? as.V : as.K) + tk * dpad + vi * 8;
          uint4 val = pf[jv];
          if (md.kv_q8) {
            // masked tokens stay zero: their codes and scale were never loaded
            const float d16 = __half2float(__ushort_as_half(pfs[jv]));
            const int8_t* cb = reinterpret_cast<const int8_t*>(&pf[jv]);
            __half hv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = __float2half_rn(d16 * static_cast<float>(cb[e]));
            val = *reinterpret_cast<uint4*>(hv);
          }
          *reinterpret_cast<uint4*>(dst) = val;
        }
      }
    };
    if (te > tb) load_tile(tb);
    for (int it = 0; it < n_iter; ++it) {
      const bool newtile = last && it == n_iter - 1;
      const int tile = tb + it;
      // ---- K/V tile (32 tokens) as fp16
      if (!newtile) {
        store_tile();
        if (tile + 1 < te) load_tile(tile + 1);
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
      math_sync();
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
      math_sync();
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
      math_sync();
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
      math_sync();
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
      math_sync();
      if (tid == 0) {
        const int key = si * hkv + kh;
        const uint32_t old = atomicAdd(&md.attn_tickets[key], 1u);
        const int is_last = old + 1u == static_cast<uint32_t>(nsplit);
        if (is_last) md.attn_tickets[key] = 0u;
        *as.flag = is_last;
      }
      math_sync();
      if (*as.flag) {
        __threadfence();
        const int item0 = sd.seq_item0[si] + kh * nsplit;
        float* wb = wbuf + warp * kMaxSplits;
        // one warp per query row: split weights over lanes, head dims over lanes
        for (int qr = warp; qr < qrows; qr += kWarps) {
          float mloc = -INFINITY;
          for (int sp = lane; sp < nsplit; sp += 32)
            mloc = fmaxf(mloc, __ldcg(md.attn_part + (static_cast<size_t>(item0 + sp) * kMaxQRows + qr) * (kMaxDh + 2) + kMaxDh));
          const float M = warp_max(mloc);
          float lloc = 0.f;
          for (int sp = lane; sp < nsplit; sp += 32) {
            const float* pp = md.attn_part + (static_cast<size_t>(item0 + sp) * kMaxQRows + qr) * (kMaxDh + 2);
            const float ms = __ldcg(pp + kMaxDh);
            const float w = ms == -INFINITY ? 0.f : expf(ms - M);
            wb[sp] = w;
            lloc = fmaf(__ldcg(pp + kMaxDh + 1), w, lloc);
          }
          const float inv = 1.0f / warp_sum(lloc);
          __syncwarp();
          float val[kMaxDh / 32];
#pragma unroll
          for (int e = 0; e < kMaxDh / 32; ++e) val[e] = 0.f;
#pragma unroll 4
          for (int sp = 0; sp < nsplit; ++sp) {
            const float w = wb[sp];
            const float* pp = md.attn_part + (static_cast<size_t>(item0 + sp) * kMaxQRows + qr) * (kMaxDh + 2);
#pragma unroll
            for (int e = 0; e < kMaxDh / 32; ++e)
              if (lane + 32 * e < dh) val[e] = fmaf(__ldcg(pp + lane + 32 * e), w, val[e]);
          }
          const int t = qr / grp, hh = kh * grp + qr % grp;
          float* o = md.o + static_cast<size_t>(row0 + t) * md.o_stride + hh * dh;
#pragma unroll
          for (int e = 0; e < kMaxDh / 32; ++e)
            if (lane + 32 * e < dh) o[lane + 32 * e] = val[e] * inv;
          __syncwarp();
        }
      }
    }
    math_sync();
  }
}

static_assert(kMaxQRows * (kMaxDh + 8) * 2 + 2 * 32 * (kMaxDh + 8) * 2 + kMaxQRows * 33 * 4 + kMaxQRows * 40 * 2 +
                      3 * kMaxQRows * 4 + 16 + kWarps * kMaxSplits * 4 <=
                  kPhaseBytes,
              "attention shared memory");
static_assert(kWarps * (2 * kMaxT * 128 + kMaxT * 10) * 4 <= kPhaseBytes, "Gated DeltaNet shared memory");

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
  math_sync();
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
// 9 warps: at most 168 registers each (three warps share a sub-partition).
__global__ void __launch_bounds__(kLaunchThreads, 1)
    mk_persistent(const ModelDesc* __restrict__ mdp, const StepDesc* __restrict__ sdp, float* attn_scratch) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int sflag;
  const Smem sm{smem_raw};
  const ModelDesc& md = *mdp;
  const StepDesc& sd = *sdp;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x < kWarps * kRing) {
    mbar_init(sm.bar(threadIdx.x / kRing, threadIdx.x % kRing), 1);
    mbar_init(sm.empty(threadIdx.x / kRing, threadIdx.x % kRing), 1);
  }
  mbar_fence_init();
  __syncthreads();
  if (warp == kWarps) {  // the producer warp
    producer_warp(md, sd, sm);
    return;
  }
  WarpCtx wc;
  wc.warp = warp;
  wc.lane = threadIdx.x & 31;
  wc.gid = blockIdx.x * kWarps + wc.warp;
  wc.c_pos = 0;

  int nbar = 0;
  float* my_scratch = attn_scratch + static_cast<size_t>(blockIdx.x) * kWarps * 2 * kMaxDh;
  // Phases: 0 embed; then per layer l: 1+5l input GEMM, 2+5l mixer,
  // 3+5l o_proj, 4+5l gate/up, 5+5l down; then lm_head; then verify.
  const int n_phases = 1 + 5 * md.n_layers + 2;
  if (md.dbg_time && blockIdx.x == 0 && threadIdx.x == 0) md.dbg_time[0] = globaltimer();
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
        if (md.layer[l].kind == MK_LAYER_GDN) gdn_phase(md, sd, l, wc, sm);
        else attn_phase(md, sd, l, sm, my_scratch);
      } else {
        gp = 4 * l + (part == 0 ? 0 : part - 1);
      }
    }
    if (gp >= 0) ok = gemm_dispatch(md, sd, gp, sm, wc);
    // a failed wait inside a phase still meets the barrier, which reports it
    const bool synced = grid_sync(md, sd, nbar, &sflag);
    if (md.dbg_time && blockIdx.x == 0 && threadIdx.x == 0) md.dbg_time[ph + 1] = globaltimer();
    if (!synced || !ok) break;
  }
}

cudaError_t launch_persistent(const ModelDesc* md, const StepDesc* sd, float* attn_scratch, int grid,
                              cudaStream_t stream) {
  void* args[] = {const_cast<ModelDesc**>(&md), const_cast<StepDesc**>(&sd), &attn_scratch};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(mk_persistent), dim3(grid), dim3(kLaunchThreads),
                                     args, kSmemBytes, stream);
}

cudaError_t configure_persistent(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(mk_persistent),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, reinterpret_cast<const void*>(mk_persistent),
                                                       kLaunchThreads, kSmemBytes);
}

}  // namespace mk
