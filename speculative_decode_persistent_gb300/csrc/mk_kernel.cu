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
#include <cuda.h>
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
  // registers only: not volatile, so the scheduler may interleave independent chains
  asm(
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
__device__ __forceinline__ float sigmoidf_(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }
__device__ __forceinline__ float siluf_(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// --------------------------------------------------------- shared memory
// The block's dynamic shared memory. Every region is addressed from this
// array directly, so the compiler keeps shared-window (32-bit) addressing in
// every phase function.
extern __shared__ __align__(128) uint8_t smem_raw[];

struct Smem {
  __device__ uint8_t* ring(int warp, int slot) const {
    return smem_raw + kOffRing + (warp * kRing + slot) * kUnitBytes;
  }
  __device__ uint64_t* bar(int warp, int slot) const {  // full: the unit has landed
    return reinterpret_cast<uint64_t*>(smem_raw + kOffBar) + warp * kRing + slot;
  }
  __device__ uint64_t* empty(int warp, int slot) const {  // the math warp is done with the slot
    return reinterpret_cast<uint64_t*>(smem_raw + kOffBar) + kWarps * kRing + warp * kRing + slot;
  }
  __device__ uint32_t* stab(int warp, int buf) const {
    return reinterpret_cast<uint32_t*>(smem_raw + kOffTab + (warp * 2 + buf) * kWarpTab);
  }
  __device__ uint8_t* act() const { return smem_raw + kOffAct; }
  __device__ float* misc() const { return reinterpret_cast<float*>(smem_raw + kOffMisc); }
  __device__ uint8_t* phase() const { return smem_raw + kOffPhase; }
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
  uint32_t c_pos;   // units consumed by this math warp
  uint32_t kv_pos;  // attention chunks consumed by this warp's group
};

// GEMM phases in step order: 4l + {0 input projections, 1 o_proj, 2 gate/up,
// 3 down} for layer l, then 4 n_layers the lm_head, then per MTP draft pass p
// six phases from mtp_gp0 + 6p: W_fc, input projections, o_proj, gate/up,
// down, and the lm_head over the draft vocabulary.
__device__ __forceinline__ int mtp_gp0(const ModelDesc& md) { return 4 * md.n_layers + 1; }

__device__ __forceinline__ const GemmDesc& gemm_desc(const ModelDesc& md, int gp) {
  const int l = gp >> 2, part = gp & 3;
  if (l < md.n_layers) {
    const LayerDesc& L = md.layer[l];
    return part == 0 ? L.in : part == 1 ? L.o : part == 2 ? L.gu : L.down;
  }
  if (gp == 4 * md.n_layers) return md.lm;
  const int q = (gp - mtp_gp0(md)) % 6;
  const LayerDesc& M = md.layer[md.n_layers];
  return q == 0 ? md.mtp_fc : q == 1 ? M.in : q == 2 ? M.o : q == 3 ? M.gu : q == 4 ? M.down : md.mtp_lm;
}

// Phases whose epilogue keeps top-1 records (the two lm_heads).
__device__ __forceinline__ bool is_top_gp(const ModelDesc& md, int gp) {
  return gp == 4 * md.n_layers || (gp > 4 * md.n_layers && (gp - mtp_gp0(md)) % 6 == 5);
}

// The attention whose KV pages are streamed right before GEMM phase gp (the
// o_proj of a gated-attention layer or of an MTP pass), as a key that grows
// along the step: layer l, or n_layers + p for draft pass p; -1 if none.
__device__ __forceinline__ int attn_key_before(const ModelDesc& md, int gp) {
  if (gp < 4 * md.n_layers) {
    const int l = gp >> 2;
    return ((gp & 3) == 1 && md.layer[l].kind == MK_LAYER_FA) ? l : -1;
  }
  if (gp <= 4 * md.n_layers) return -1;
  const int q = gp - mtp_gp0(md);
  return q % 6 == 2 ? md.n_layers + q / 6 : -1;
}

__device__ __forceinline__ Assign assign_for(const GemmDesc& g, int R, int grid, int cta, int warp) {
  return assign_units(g.n_tiles, g.nsb, R, grid, cta, warp);
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
  // the step's accumulation buffers start at zero: first input projections,
  // first gate/up, lm_head
  {
    const int stride = gridDim.x * kThreads, t0 = blockIdx.x * kThreads + threadIdx.x;
    for (int idx = t0; idx < sd.R * md.n_in_max; idx += stride) md.yin[idx] = 0.f;
    for (int idx = t0; idx < sd.R * 2 * md.F; idx += stride) md.gu[idx] = 0.f;
    for (int idx = t0; idx < sd.R * md.V; idx += stride) md.logits[idx] = 0.f;
  }
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
      const float xv = ds * static_cast<float>(q) - dm;
      md.x[static_cast<size_t>(r) * md.H + sb * 256 + 32 * j + i] = xv;
    }
  }
}

// --------------------------------------------------------- GEMM prologue
// Fills the activation region for reduction slice [sb0, sb0 + nsb_s): for each
// row r, column 2r holds the fp16 high part and column 2r+1 the low part of the
// input vector, each column in the per-32 permuted order of the B fragments;
// then sx[sb][j][r] (rows padded to kSxStride) = sum of (high + low) over
// sub-block j. Loads are float4,
// and per-row norms reduce over the whole block in a fixed order.
__device__ __forceinline__ int act_perm(int kl) {
  const int i = kl & 31;
  const int ks_in = i >> 4, rr = i & 15;
  const int c = (rr & 7) >> 1, half = rr >> 3, e = rr & 1;
  return (kl & ~31) + c * 8 + ks_in * 4 + half * 2 + e;
}

__device__ __forceinline__ void put_act(__half* act, int cs2, int R, float* sx, int r, int kl, const float (&u)[4],
                                        int lane) {
  // packed conversions: high = fp16(u), low = fp16(u - high)
  const __half2 h01 = __floats2half2_rn(u[0], u[1]), h23 = __floats2half2_rn(u[2], u[3]);
  const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
  const __half2 l01 = __floats2half2_rn(u[0] - f01.x, u[1] - f01.y);
  const __half2 l23 = __floats2half2_rn(u[2] - f23.x, u[3] - f23.y);
  // the sub-block sums feed only the Q4 min term: the fp32 values differ
  // from high + low by at most 2^-22 relative
  float part = (u[0] + u[1]) + (u[2] + u[3]);
  // k and k+1 (and k+2, k+3) are adjacent pairs in the permuted order
  const int p0 = act_perm(kl), p2 = act_perm(kl + 2);
  __half* chi = act + (2 * r) * cs2;
  __half* clo = act + (2 * r + 1) * cs2;
  *reinterpret_cast<__half2*>(chi + p0) = h01;
  *reinterpret_cast<__half2*>(chi + p2) = h23;
  *reinterpret_cast<__half2*>(clo + p0) = l01;
  *reinterpret_cast<__half2*>(clo + p2) = l23;
  // 8 consecutive threads hold one 32-wide sub-block
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  part += __shfl_xor_sync(0xffffffffu, part, 4);
  if ((lane & 7) == 0) sx[((kl >> 8) * 8 + ((kl & 255) >> 5)) * kSxStride + r] = part;
}

// One round of loads: every thread issues all of its source float4 loads
// (up to kB groups) before using any of them, so the prologue costs about
// one L2 round trip (plus the row norms' batches for an RMSNorm).
// Gated DeltaNet output: each head's 128 (or 64) values are the float4s of
// 32 (or 16) consecutive lanes, so its norm is a shuffle sum.
// One prologue kind's rounds, as its own straight-line code: a phase runs one
// kind, so the instructions it executes are contiguous.
template <int PRO>
__device__ __forceinline__ void prologue_rounds(const ModelDesc& md, const GemmDesc& g, int R, int k0, int per_row,
                                                __half* act, int cs2, float* sx, float* red) {
  constexpr int kB = 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = R * per_row;
  for (int base = 0; base < total; base += kThreads * kB) {
    // every source of this round, norm gains included, is loaded before any is used
    float4 s1[kB], s2[kB], s3[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int idx = base + b * kThreads + tid;
      s1[b] = s2[b] = s3[b] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < total) {
        const int r = idx / per_row, k = k0 + (idx - r * per_row) * 4;
        if constexpr (PRO == PRO_RMS_X) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.x + static_cast<size_t>(r) * md.H + k));
          s2[b] = *reinterpret_cast<const float4*>(g.gain + k);
        } else if constexpr (PRO == PRO_GDN_OUT) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.o + static_cast<size_t>(r) * md.o_stride + k));
          s2[b] = __ldcg(reinterpret_cast<const float4*>(md.yin + static_cast<size_t>(r) * md.n_in_max + md.conv_ch + k));
          s3[b] = *reinterpret_cast<const float4*>(g.gain + k % md.dv);
        } else if constexpr (PRO == PRO_FA_OUT) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.o + static_cast<size_t>(r) * md.o_stride + k));
          s2[b] = __ldcg(reinterpret_cast<const float4*>(md.yin + static_cast<size_t>(r) * md.n_in_max + md.hq * md.dh + k));
        } else if constexpr (PRO == PRO_MTP_IN) {
          s1[b] = __ldcg(reinterpret_cast<const float4*>(md.mtp_in + static_cast<size_t>(r) * 2 * md.H + k));
        } else {  // SwiGLU of the gate/up pair: 4 consecutive f share one 8-row block
          const float* gr = md.gu + static_cast<size_t>(r) * 2 * md.F + (k >> 3) * 16 + (k & 7);
          s1[b] = __ldcg(reinterpret_cast<const float4*>(gr));
          s2[b] = __ldcg(reinterpret_cast<const float4*>(gr + 8));
        }
      }
    }
    if constexpr (PRO == PRO_RMS_X) {
      // this slice's sums of squares per row: the 32 float4 of one warp's
      // load b lie in one row (a row holds a multiple of 64 float4)
#pragma unroll
      for (int b = 0; b < kB; ++b) {
        const int idx0 = base + b * kThreads + warp * 32;
        if (idx0 < total) {
          float sq = fmaf(s1[b].x, s1[b].x, fmaf(s1[b].y, s1[b].y, fmaf(s1[b].z, s1[b].z, s1[b].w * s1[b].w)));
          sq = warp_sum(sq);
          if (lane == 0) red[warp * kMaxRows + idx0 / per_row] += sq;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int idx = base + b * kThreads + tid;
      if (idx < total) {  // warp-uniform: total is a multiple of 64
        const int r = idx / per_row, kl = (idx - r * per_row) * 4, k = k0 + kl;
        float u[4];
        if constexpr (PRO == PRO_RMS_X) {  // x (.) gain; the row's 1/rms scales the GEMM's outputs
          const float4 gg = s2[b];
          u[0] = s1[b].x * gg.x; u[1] = s1[b].y * gg.y; u[2] = s1[b].z * gg.z; u[3] = s1[b].w * gg.w;
        } else if constexpr (PRO == PRO_GDN_OUT) {
          float hs = fmaf(s1[b].x, s1[b].x, fmaf(s1[b].y, s1[b].y, fmaf(s1[b].z, s1[b].z, s1[b].w * s1[b].w)));
          for (int off = 1; off < md.dv / 4; off <<= 1) hs += __shfl_xor_sync(0xffffffffu, hs, off);
          const float sc = 1.0f / sqrtf(hs / static_cast<float>(md.dv) + md.eps);
          const float4 gg = s3[b];
          u[0] = s1[b].x * sc * gg.x * siluf_(s2[b].x); u[1] = s1[b].y * sc * gg.y * siluf_(s2[b].y);
          u[2] = s1[b].z * sc * gg.z * siluf_(s2[b].z); u[3] = s1[b].w * sc * gg.w * siluf_(s2[b].w);
        } else if constexpr (PRO == PRO_FA_OUT) {
          u[0] = s1[b].x * sigmoidf_(s2[b].x); u[1] = s1[b].y * sigmoidf_(s2[b].y);
          u[2] = s1[b].z * sigmoidf_(s2[b].z); u[3] = s1[b].w * sigmoidf_(s2[b].w);
        } else if constexpr (PRO == PRO_MTP_IN) {
          u[0] = s1[b].x; u[1] = s1[b].y; u[2] = s1[b].z; u[3] = s1[b].w;
        } else {
          u[0] = siluf_(s1[b].x) * s2[b].x; u[1] = siluf_(s1[b].y) * s2[b].y;
          u[2] = siluf_(s1[b].z) * s2[b].z; u[3] = siluf_(s1[b].w) * s2[b].w;
          if (md.dbg_logits)  // debug outputs on: keep the SwiGLU rows for mk_debug_scratch
            *reinterpret_cast<float4*>(md.h + static_cast<size_t>(r) * md.F + k) = make_float4(u[0], u[1], u[2], u[3]);
        }
        put_act(act, cs2, R, sx, r, kl, u, lane);
      }
    }
  }
}

constexpr int kTopRecOffFloats = 640;  // per-warp top-1 records inside misc (floats)
// Per-warp 1/rms of the rows of an RMSNorm GEMM phase, inside misc (floats).
constexpr int kInvOff = 840;
static_assert(kInvOff >= kTopRecOffFloats + kWarps * 2 * kMaxRows && (kInvOff + kWarps * kMaxRows) * 4 <= kAttnBarOff,
              "RMSNorm scales in misc");

// The activation operand of one GEMM phase for this block's reduction slice.
// An RMSNorm phase feeds x (.) gain and leaves the row's 1/rms to scale the
// GEMM's outputs (it is one factor per row): with one slice the block's own
// loads are the whole row, so each warp takes the block's sums of squares;
// with several, the slice's first block publishes its partial sums and each
// warp adds the partials of all slices (load_inv) before its first output.
template <int NT>
__device__ void gemm_prologue(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g, int gp, const Assign& a,
                              const Smem& sm) {
  const int R = sd.R;
  const int k0 = a.sb0 * 256, ks = a.nsb_s * 256;
  const int cstride = act_col_stride(a.nsb_s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __half* act = reinterpret_cast<__half*>(sm.act());
  float* sx = reinterpret_cast<float*>(sm.act() + 2 * R * cstride);
  float* misc = sm.misc();
  float* red = misc + 512;  // [warp][row] sums of squares of this slice (RMSNorm phases)
  const int per_row = ks / 4;
  const int cs2 = cstride / 2;
  if (g.pro == PRO_RMS_X) {
    if (lane < kMaxRows) red[warp * kMaxRows + lane] = 0.f;
    __syncwarp();
  }
  switch (g.pro) {
    case PRO_RMS_X: prologue_rounds<PRO_RMS_X>(md, g, R, k0, per_row, act, cs2, sx, red); break;
    case PRO_GDN_OUT: prologue_rounds<PRO_GDN_OUT>(md, g, R, k0, per_row, act, cs2, sx, red); break;
    case PRO_FA_OUT: prologue_rounds<PRO_FA_OUT>(md, g, R, k0, per_row, act, cs2, sx, red); break;
    case PRO_MTP_IN: prologue_rounds<PRO_MTP_IN>(md, g, R, k0, per_row, act, cs2, sx, red); break;
    default: prologue_rounds<PRO_H>(md, g, R, k0, per_row, act, cs2, sx, red); break;
  }
  math_sync();
  if (g.pro == PRO_RMS_X) {
    float tot = 0.f;
    if (lane < R)
      for (int w = 0; w < kWarps; ++w) tot += red[w * kMaxRows + lane];
    if (a.sc.S == 1) {
      if (lane < R) misc[kInvOff + warp * kMaxRows + lane] = 1.0f / sqrtf(tot / static_cast<float>(md.H) + md.eps);
    } else if (static_cast<int>(blockIdx.x) == a.cta0 && warp == 0) {
      if (lane < R) md.norm_part[(static_cast<size_t>(gp) * kMaxNormSlices + a.sl) * kMaxRows + lane] = tot;
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(md.norm_cnt + gp) : "memory");
      }
    }
    __syncwarp();
  }
}

// A warp's 1/rms of the rows of a sliced RMSNorm phase: a bounded wait until
// every slice has published its partial sums of squares, then their sum in
// slice order. False (and the error word set) on timeout or another error.
__device__ __noinline__ bool load_inv(const ModelDesc& md, const StepDesc& sd, int gp, int S, int warp, int lane) {
  int ok = 1;
  if (lane == 0) {
    volatile int32_t* err = md.err;
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire(md.norm_cnt + gp) >= static_cast<uint32_t>(S)) break;
      if ((it & 15u) == 15u) {
        if (*err != 0) { ok = 0; break; }
        const uint64_t now = globaltimer();
        if (t0 == 0) t0 = now;
        else if (now - t0 > sd.barrier_timeout_ns || it > (1u << 30)) {
          atomicCAS(md.err, 0, DEV_BARRIER_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  if (lane < sd.R) {
    (void)ld_acquire(md.norm_cnt + gp);  // this lane's own acquire of the published sums
    float tot = 0.f;
    for (int sl = 0; sl < S; ++sl) tot += __ldcg(md.norm_part + (static_cast<size_t>(gp) * kMaxNormSlices + sl) * kMaxRows + lane);
    reinterpret_cast<float*>(smem_raw + kOffMisc)[kInvOff + warp * kMaxRows + lane] =
        1.0f / sqrtf(tot / static_cast<float>(md.H) + md.eps);
  }
  __syncwarp();
  return true;
}

// ------------------------------------------------------------- top-1 state
// Larger value wins; on an exact tie the lower vocabulary index wins.
__device__ __forceinline__ void top1_merge(float& a1, int& ai, float b1, int bi) {
  if (b1 > a1 || (b1 == a1 && bi < ai)) {
    a1 = b1;
    ai = bi;
  }
}

// Running top-1 of every row over the lm_head tiles a warp has finished:
// kMaxRows (value, index) pairs per warp in the misc region.
constexpr int kTopRecOff = kTopRecOffFloats;  // float offset inside misc
static_assert((kTopRecOff + kWarps * 2 * kMaxRows) * 4 <= kAttnBarOff, "top-1 records");
__device__ __forceinline__ float* top_rec(int warp) {
  return reinterpret_cast<float*>(smem_raw + kOffMisc) + kTopRecOff + warp * 2 * kMaxRows;
}

// --------------------------------------------------------- GEMM epilogue
// v[r] is the complete output of the lane's row n = 32 tile + lane for
// activation row r. For a tile that several warps computed, the outputs were
// summed in global memory (red.add into the phase's output buffer) and v was
// read back from there: `summed` marks that case (then the stores need
// nothing more). Residual adds never come here: every warp red.adds its part.
template <int NT, bool TOP>
__device__ __forceinline__ void gemm_epilogue(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g,
                                              uint32_t tile, const float (&v)[4 * NT], int lane, int warp,
                                              bool summed) {
  const int R = sd.R;
  const int n = static_cast<int>(tile) * kTileRows + lane;
  switch (g.epi) {
    case EPI_STORE_YIN:
      if (!summed && n < g.n_out) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) md.yin[static_cast<size_t>(r) * md.n_in_max + n] = v[r];
      }
      break;
    case EPI_RESID_X:  // added into x by red.add in the flush; nothing completes here
      break;
    case EPI_STORE_GU:
      if (!summed && n < g.n_out) {
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) md.gu[static_cast<size_t>(r) * 2 * md.F + n] = v[r];
      }
      break;
    case EPI_TOP2:
      if (TOP) {
        float* rec = top_rec(warp);
#pragma unroll
        for (int r = 0; r < 4 * NT; ++r)
          if (r < R) {
            float x = -FLT_MAX;
            int ix = 0x7fffffff;
            if (n < g.n_out) {
              x = v[r];
              ix = n;
              if (!isfinite(x)) atomicOr(&md.err[1], 1);
              if (md.dbg_logits && g.dump) md.dbg_logits[static_cast<size_t>(r) * md.V + n] = x;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float ox = __shfl_xor_sync(0xffffffffu, x, o);
              const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
              top1_merge(x, ix, ox, oi);
            }
            if (lane == 0) {
              float b = rec[2 * r];
              int bi = __float_as_int(rec[2 * r + 1]);
              top1_merge(b, bi, x, ix);
              rec[2 * r] = b;
              rec[2 * r + 1] = __int_as_float(bi);
            }
          }
        __syncwarp();
      }
      break;
  }
}

// ------------------------------------------------------------- GEMM phase
// The math warp may read ring position `pos`: a try-wait on its full barrier,
// then (rarely) the bounded wait. Inline, so the unit loop makes no call.
__device__ __forceinline__ bool wait_slot(const Smem& sm, int warp, uint32_t pos, const ModelDesc& md,
                                          uint64_t timeout_ns) {
  uint64_t* b = sm.bar(warp, pos % kRing);
  const uint32_t parity = (pos / kRing) & 1u;
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  volatile int32_t* err = md.err;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*err != 0) return false;
      if (globaltimer() - t0 > timeout_ns || it > (1u << 26)) {
        atomicCAS(md.err, 0, DEV_COPY_TIMEOUT);
        return false;
      }
    }
  }
}

// One finished tile segment of an lm_head phase (top-1 records, optional
// debug dump, completion tickets), out of line: row `lane` of the segment's
// outputs for every activation row is in stage[lane * 17 + r], already
// scaled by the rows' 1/rms. A tile the warp computed whole goes straight to
// its epilogue; a split one is summed by red.add into the logits buffer, and
// when the reduction is not sliced the last contributor (completion ticket)
// runs the epilogue on the sum.
template <int NT, bool TOP>
__device__ __noinline__ void tile_out_top(const ModelDesc& md, const StepDesc& sd, int gp, uint32_t tile, bool whole,
                                          const float* stage, int lane, int warp) {
  const GemmDesc& g = gemm_desc(md, gp);
  const int R = sd.R;
  float v[4 * NT];
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r) v[r] = r < R ? stage[lane * 17 + r] : 0.f;
  __syncwarp();
  if (whole) {
    gemm_epilogue<NT, TOP>(md, sd, g, tile, v, lane, warp, false);
    return;
  }
  float* dst = md.logits;
  const int dstride = md.V;
  const int n = static_cast<int>(tile) * kTileRows + lane;
  if (n < g.n_out) {
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r)
      if (r < R) atomicAdd(dst + static_cast<size_t>(r) * dstride + n, v[r]);
  }
  // sliced logits are scanned by lm_argmax after the next barrier
  const Sched sc = make_sched(g.nsb, R);
  if (sc.S > 1) return;
  __threadfence();
  __syncwarp();
  uint32_t last = 0;
  if (lane == 0) {
    const uint32_t na = tile_arrivals(sc, g.n_tiles, g.nsb, gridDim.x, tile);
    const uint32_t old = atomicAdd(&md.tickets[tile], 1u);
    last = (old + 1u == na) ? 1u : 0u;
    if (last) md.tickets[tile] = 0u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
#pragma unroll
  for (int r = 0; r < 4 * NT; ++r)
    v[r] = (r < R && n < g.n_out) ? __ldcg(dst + static_cast<size_t>(r) * dstride + n) : 0.f;
  gemm_epilogue<NT, TOP>(md, sd, g, tile, v, lane, warp, true);
}

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


// A 6-bit field as an exact float without a conversion instruction: its bits
// become the low mantissa bits of 2^23, which is then subtracted.
__device__ __forceinline__ float u6f(uint32_t v) { return __uint_as_float(0x4B000000u | v) - 8388608.0f; }

// One step of the own-row header decode: sub-block j of the lane's row in
// the next unit -> its fp32 scale d * sc_j * 2^24 (or 2^20), exact, into the
// scale table, and the min term dmin * m_j * sum_j(x) added into mtmp (four
// activation rows per 16-byte load of the padded sub-block sums).
template <int NT>
__device__ __forceinline__ float decode_step(int j, const uint4& hdr, float dscale, float dmin, const float* sxb,
                                             float (&mtmp)[4 * NT]) {
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
  const float dm = dmin * u6f(m);  // exact: 11-bit x 6-bit
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float4 sv = *reinterpret_cast<const float4*>(sxb + j * kSxStride + 4 * i);
    mtmp[4 * i + 0] = fmaf(dm, sv.x, mtmp[4 * i + 0]);
    mtmp[4 * i + 1] = fmaf(dm, sv.y, mtmp[4 * i + 1]);
    mtmp[4 * i + 2] = fmaf(dm, sv.z, mtmp[4 * i + 2]);
    mtmp[4 * i + 3] = fmaf(dm, sv.w, mtmp[4 * i + 3]);
  }
  return dscale * u6f(sc);  // exact: 11-bit x 6-bit
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
  if (g.zero_buf != ZERO_NONE) {  // a later phase's accumulation buffer starts at zero
    float* zp = g.zero_buf == ZERO_GU ? md.gu : md.yin;
    const int cols = g.zero_buf == ZERO_GU ? 2 * md.F : md.n_in_max;
    for (int idx = blockIdx.x * kThreads + threadIdx.x; idx < R * cols; idx += grid * kThreads) zp[idx] = 0.f;
  }
  gemm_prologue<NT>(md, sd, g, gp, a, sm);

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
  if (TOP) {
    float* rec = top_rec(wc.warp);
    if (lane < R) {
      rec[2 * lane] = -FLT_MAX;
      rec[2 * lane + 1] = __int_as_float(0x7fffffff);
    }
    __syncwarp();
  }

  float acc[2][NT][4];
  float mn[4 * NT], mtmp[4 * NT];
#pragma unroll
  for (int rb = 0; rb < 2; ++rb)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rb][nt][e] = 0.f;

  // where this phase's outputs go (stores of whole tiles, red.add of split ones)
  float* const dst = g.epi == EPI_STORE_YIN ? md.yin : g.epi == EPI_RESID_X ? md.x : md.gu;
  const int dstride = g.epi == EPI_STORE_YIN ? md.n_in_max : g.epi == EPI_RESID_X ? md.H : 2 * md.F;
  const bool rms = g.pro == PRO_RMS_X;
  bool ok = true;
  bool inv_ready = !rms || a.sc.S == 1;
  if (a.u1 > a.u0) {
    uint32_t tile = a.u0 / nsb_s;
    int sbl = static_cast<int>(a.u0 - tile * nsb_s);
    uint32_t seg_u0 = a.u0;
    // pipeline fill: the first unit's own-row scales into table 0, its min term into mn
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) mtmp[r] = 0.f;
    if (!wait_slot(sm, wc.warp, wc.c_pos, md, sd.barrier_timeout_ns)) {
      ok = false;
    } else {
      const uint4 hdr = *reinterpret_cast<const uint4*>(sm.ring(wc.warp, wc.c_pos % kRing) + 16 * lane);
      const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
      const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
      float scl[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) scl[j] = decode_step<NT>(j, hdr, d * row_unscale, dmin, sx + sbl * 8 * kSxStride, mtmp);
      store_scales(reinterpret_cast<float*>(sm.stab(wc.warp, 0)), scl, og, orb, ohi);
    }
#pragma unroll
    for (int r = 0; r < 4 * NT; ++r) mn[r] = mtmp[r];
    __syncwarp();
    for (uint32_t u = a.u0; ok && u < a.u1; ++u) {
      const int cur = static_cast<int>((u - a.u0) & 1u);
      const bool has_next = u + 1 < a.u1;
      if (has_next && !wait_slot(sm, wc.warp, wc.c_pos + 1, md, sd.barrier_timeout_ns)) { ok = false; break; }
      const uint8_t* unit = sm.ring(wc.warp, wc.c_pos % kRing);
      // the next unit's header (the current one's when this is the last: decoded, never used)
      const uint4 hdrn =
          *reinterpret_cast<const uint4*>(sm.ring(wc.warp, (wc.c_pos + (has_next ? 1u : 0u)) % kRing) + 16 * lane);
      const float dscalen = __half2float(__ushort_as_half(static_cast<unsigned short>(hdrn.x & 0xffffu))) * row_unscale;
      const float dminn = __half2float(__ushort_as_half(static_cast<unsigned short>(hdrn.x >> 16)));
      const int sbl_next = sbl + 1 == nsb_s ? 0 : sbl + 1;
      const float* tab = reinterpret_cast<const float*>(sm.stab(wc.warp, cur));
      float* tabn = reinterpret_cast<float*>(sm.stab(wc.warp, cur ^ 1));
#pragma unroll
      for (int r = 0; r < 4 * NT; ++r) mtmp[r] = 0.f;
      const uint8_t* codes = unit + kUnitHdr + lane * 16;
      const int boff = sbl * 512;
      const float* sxn = sx + sbl_next * 8 * kSxStride;
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
        uint32_t av[4];
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {  // rows 16rb..16rb+15: words x/z (rb 0) or y/w (rb 1)
          float t[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) t[nt][e] = 0.f;
          dequant_word(rb ? w4.y : w4.x, av);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(t[nt], av[0], av[1], av[2], av[3], bf[nt].x, bf[nt].y);
          dequant_word(rb ? w4.w : w4.z, av);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(t[nt], av[0], av[1], av[2], av[3], bf[nt].z, bf[nt].w);
          const float sa = rb ? s4.z : s4.x, sb = rb ? s4.w : s4.y;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[rb][nt][0] = fmaf(sa, t[nt][0], acc[rb][nt][0]);
            acc[rb][nt][1] = fmaf(sa, t[nt][1], acc[rb][nt][1]);
            acc[rb][nt][2] = fmaf(sb, t[nt][2], acc[rb][nt][2]);
            acc[rb][nt][3] = fmaf(sb, t[nt][3], acc[rb][nt][3]);
          }
        }
        scl[kp] = decode_step<NT>(kp, hdrn, dscalen, dminn, sxn, mtmp);
      }
      store_scales(tabn, scl, og, orb, ohi);
      release_unit(wc, sm);  // includes __syncwarp: both tables are settled
      if (++sbl == nsb_s || u + 1 == a.u1) {
        // the tile segment ends: transpose the warp's outputs through the
        // table just consumed (row = lane), subtract the min term, scale an
        // RMSNorm phase's rows by their 1/rms, and store or red.add them
        float* stage = reinterpret_cast<float*>(sm.stab(wc.warp, cur));
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int r = nt * 4 + cq;
            if (r < R) {
              stage[(rb * 16 + gq) * 17 + r] = acc[rb][nt][0] + acc[rb][nt][1];
              stage[(rb * 16 + gq + 8) * 17 + r] = acc[rb][nt][2] + acc[rb][nt][3];
            }
          }
        if (!inv_ready) {  // a sliced RMSNorm phase: every slice's row sums, once
          if (!load_inv(md, sd, gp, a.sc.S, wc.warp, lane)) { ok = false; break; }
          inv_ready = true;
        }
        __syncwarp();
        const uint32_t tu0 = tile * nsb_s;
        const bool whole = a.sc.S == 1 && seg_u0 == tu0 && u + 1 == tu0 + nsb_s && g.epi != EPI_RESID_X;
        const float* inv = reinterpret_cast<const float*>(smem_raw + kOffMisc) + kInvOff + wc.warp * kMaxRows;
        if (TOP) {
#pragma unroll
          for (int r = 0; r < 4 * NT; ++r)
            if (r < R) stage[lane * 17 + r] = (stage[lane * 17 + r] - mn[r]) * inv[r];
          __syncwarp();
          tile_out_top<NT, TOP>(md, sd, gp, tile, whole, stage, lane, wc.warp);
        } else {
          const int n = static_cast<int>(tile) * kTileRows + lane;
          if (n < g.n_out) {
#pragma unroll
            for (int r = 0; r < 4 * NT; ++r)
              if (r < R) {
                float vr = stage[lane * 17 + r] - mn[r];
                if (rms) vr *= inv[r];
                float* p = dst + static_cast<size_t>(r) * dstride + n;
                if (whole) *p = vr;
                else atomicAdd(p, vr);
              }
          }
          __syncwarp();
        }
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

  if (TOP && lane < R) {  // one record per warp and row
    const float* rec = top_rec(wc.warp);
    md.top_val[static_cast<size_t>(wc.gid) * kMaxRows + lane] = rec[2 * lane];
    md.top_idx[static_cast<size_t>(wc.gid) * kMaxRows + lane] = __float_as_int(rec[2 * lane + 1]);
  }
  return ok;
}

__device__ __forceinline__ bool gemm_dispatch(const ModelDesc& md, const StepDesc& sd, int gp, const Smem& sm,
                                              WarpCtx& wc) {
  const bool top = is_top_gp(md, gp);
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
    // causal conv + SiLU of channel ch at row t; when `hist_out` the channel's
    // history after row t (inputs t-2, t-1, t) goes straight to that row's
    // state slot from the values already loaded
    auto conv = [&](int ch, int t, bool hist_out) -> float {
      const float4 w = *reinterpret_cast<const float4*>(cw + ch * 4);
      const float p0 = pre(ch, t - 3), p1 = pre(ch, t - 2), p2 = pre(ch, t - 1), p3 = pre(ch, t);
      if (hist_out && (sd.seq_snap_all[si] || t == T - 1)) {
        const size_t ss = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_out[si][t];
        float* ho = md.conv_state + (ss * md.n_gdn + gi) * 3 * C + ch;
        __stcg(ho, p1);
        __stcg(ho + C, p2);
        __stcg(ho + 2 * C, p3);
      }
      return siluf_(fmaf(w.w, p3, fmaf(w.z, p2, fmaf(w.y, p1, w.x * p0))));
    };
    // q/k history is written once per qk head: by the tasks of its first
    // v-head, each for its own 8 channels of q and of k
    const bool qk_owner = h % (hv / hk) == 0;
    // normalised q, k of this head for every row: [t][dk] each, per warp
    float* qs = reinterpret_cast<float*>(sm.phase()) + wc.warp * (2 * kMaxT * 128 + kMaxT * 10);
    float* ks = qs + kMaxT * 128;
    // per-row gates and this task's 8 v values: [t] in shared memory after q, k
    float* vs = ks + kMaxT * 128;  // [kMaxT][8]
    float* gs = vs + kMaxT * 8;    // [kMaxT][2] alpha, beta
    if (T == 1) {
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
              const bool own = qk_owner && d >= i0 && d < i0 + 8;
              q4[e] = conv(g * dk + d, t, own);
              k4[e] = conv(hk * dk + g * dk + d, t, own);
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
          if (lane < 8) vs[t * 8 + lane] = conv(2 * hk * dk + h * dv + i0 + lane, t, true);
          if (lane == 0) {
            const float* yr = md.yin + static_cast<size_t>(row0 + t) * md.n_in_max;
            gs[t * 2 + 0] = sigmoidf_(__ldcg(yr + a_off + h));
            gs[t * 2 + 1] = sigmoidf_(__ldcg(yr + b_off + h));
          }
        }
      }
    } else {
      // T > 1: each channel's inputs are one sliding window over the history
      // and the sequence's rows
      const bool snap_rows = sd.seq_snap_all[si] != 0;
      auto hist_store = [&](int ch, int t, float a, float b, float c) {
        if (snap_rows || t == T - 1) {
          const size_t ss = static_cast<size_t>(seq) * md.n_slots + sd.seq_slot_out[si][t];
          float* ho = md.conv_state + (ss * md.n_gdn + gi) * 3 * C + ch;
          __stcg(ho, a);
          __stcg(ho + C, b);
          __stcg(ho + 2 * C, c);
        }
      };
      // each channel's inputs are loaded once as a sliding window over the
      // history and the sequence's rows; every row's conv then comes from registers
      float sq[kMaxT], sk[kMaxT];
  #pragma unroll
      for (int t = 0; t < kMaxT; ++t) sq[t] = sk[t] = 0.f;
  #pragma unroll 1
      for (int e = 0; e < 4; ++e) {
        if (e < ne) {
          const int d = lane + 32 * e;
          const int chq = g * dk + d, chk = hk * dk + g * dk + d;
          const bool own = qk_owner && d >= i0 && d < i0 + 8;
          const float4 wq = *reinterpret_cast<const float4*>(cw + chq * 4);
          const float4 wk = *reinterpret_cast<const float4*>(cw + chk * 4);
          float xq[kMaxT + 3], xk[kMaxT + 3];
  #pragma unroll
          for (int j = 0; j < kMaxT + 3; ++j) {
            xq[j] = xk[j] = 0.f;
            if (j < T + 3) {
              xq[j] = pre(chq, j - 3);
              xk[j] = pre(chk, j - 3);
            }
          }
  #pragma unroll
          for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
              const float q = siluf_(fmaf(wq.w, xq[t + 3], fmaf(wq.z, xq[t + 2], fmaf(wq.y, xq[t + 1], wq.x * xq[t]))));
              const float k = siluf_(fmaf(wk.w, xk[t + 3], fmaf(wk.z, xk[t + 2], fmaf(wk.y, xk[t + 1], wk.x * xk[t]))));
              qs[t * 128 + d] = q;
              ks[t * 128 + d] = k;
              sq[t] = fmaf(q, q, sq[t]);
              sk[t] = fmaf(k, k, sk[t]);
              if (own) {
                hist_store(chq, t, xq[t + 1], xq[t + 2], xq[t + 3]);
                hist_store(chk, t, xk[t + 1], xk[t + 2], xk[t + 3]);
              }
            }
          }
        }
      }
      if (lane < 8) {
        const int chv = 2 * hk * dk + h * dv + i0 + lane;
        const float4 wv = *reinterpret_cast<const float4*>(cw + chv * 4);
        float xv[kMaxT + 3];
  #pragma unroll
        for (int j = 0; j < kMaxT + 3; ++j) xv[j] = j < T + 3 ? pre(chv, j - 3) : 0.f;
  #pragma unroll
        for (int t = 0; t < kMaxT; ++t)
          if (t < T) {
            vs[t * 8 + lane] = siluf_(fmaf(wv.w, xv[t + 3], fmaf(wv.z, xv[t + 2], fmaf(wv.y, xv[t + 1], wv.x * xv[t]))));
            hist_store(chv, t, xv[t + 1], xv[t + 2], xv[t + 3]);
          }
      }
      if (lane < T) {
        const float* yr = md.yin + static_cast<size_t>(row0 + lane) * md.n_in_max;
        gs[lane * 2 + 0] = sigmoidf_(__ldcg(yr + a_off + h));
        gs[lane * 2 + 1] = sigmoidf_(__ldcg(yr + b_off + h));
      }
      // L2 norms of q and k per row
  #pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < T) {
          const float iq = 1.0f / sqrtf(warp_sum(sq[t]) + md.eps), ik = 1.0f / sqrtf(warp_sum(sk[t]) + md.eps);
  #pragma unroll
          for (int e = 0; e < 4; ++e)
            if (e < ne) {
              qs[t * 128 + lane + 32 * e] *= iq;
              ks[t * 128 + lane + 32 * e] *= ik;
            }
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
    __syncwarp();
  }
}

// ---------------------------------------------------------------- attention
// Split-K flash decoding over the paged KV pool for one (sequence, kv head,
// split): all T x (hq/hkv) query rows of the kv head share every K/V page.
// The last split also RoPEs, rounds or quantises and appends this step's own
// keys and values, then attends to them with the causal mask across the draft
// rows. Splits write (m, l, acc) partials; once all of a (sequence, head)'s
// splits have announced theirs, every split block merges its share.
//
// The mma work is transposed so that the head dimension and the tokens are
// the mma's M and K: per 16-token chunk, S^T = K Q^T (16 tokens x 8 query
// rows per n-tile) and O^T += V^T P^T (head dims x 8 rows). A group of warps
// takes one or two chunks per step; each warp owns a share of the head dims
// for every n-tile (its S^T share, its O^T rows), the shares meet in shared
// memory, one owner warp per n-tile takes the online-softmax step and hands
// back P^T, with two named-barrier syncs of the group per step. Pages arrive
// by tensor copies issued by the producer warp into staging slots (the
// weight ring, idle during attention). The step's own rows form one more
// chunk (causal), built by the last split.
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Two bytes of x = w ^ 0x80808080 (selected by sel) -> the binary16 pair of
// the original signed bytes, exactly: (byte + 128) becomes the mantissa of
// 1024.0, then 1152.0 is subtracted.
__device__ __forceinline__ uint32_t s8x2_to_h2(uint32_t x, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x64646464u), "r"(sel));
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&r), __half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return h2u(h);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Byte offset, inside one K (or V) box set of a slot, of byte b of token t.
__device__ __forceinline__ int kv_off(const AttnSlot& L, int t, int b) {
  const int bx = b / L.box_w, bb = b - bx * L.box_w;
  const int base = bx * kChunk * L.box_w + t * L.box_w;
  return L.swz ? base + ((((bb >> 4) ^ (t & 7)) << 4) | (bb & 15)) : base + bb;
}

struct AttnBuf {
  uint8_t* slots;   // first slot, 1024-byte aligned inside the ring region
  uint64_t* full;   // [kAttnMaxSlots]: the chunk has landed
  uint64_t* empty;  // [kAttnMaxSlots]: every warp of the group is done with it
};

__device__ __forceinline__ AttnBuf attn_buf(const Smem& sm) {
  AttnBuf b;
  const uint32_t a = smem_u32(smem_raw + kOffRing);
  b.slots = smem_raw + kOffRing + ((1024u - (a & 1023u)) & 1023u);
  b.full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sm.misc()) + kAttnBarOff);
  b.empty = b.full + kAttnMaxSlots;
  return b;
}

struct AttnItem {
  int si, kh, j, nsplit, cb, nch;
};

// Item = (sequence, kv head, split); split j covers chunks [cb, cb + nch).
__device__ __forceinline__ AttnItem attn_item(const StepDesc& sd, int hkv, int item) {
  AttnItem it;
  int si = 0;
  while (si + 1 < sd.n_seq && item >= sd.seq_item0[si + 1]) ++si;
  const int local = item - sd.seq_item0[si];
  it.si = si;
  it.nsplit = sd.seq_nsplit[si];
  it.kh = local / it.nsplit;
  it.j = local % it.nsplit;
  const int nchunk = (sd.seq_len[si] + kChunk - 1) / kChunk;
  const int cps = sd.seq_chunks_per_split[si];
  it.cb = it.j * cps;
  it.nch = max(0, min(nchunk, it.cb + cps) - it.cb);
  return it;
}

// Producer side: lane tg < ng walks group tg's chunks of this block's items
// (chunk i of an item belongs to group i % ng) and copies each page (K and V
// boxes, and the q8 scales) into the group's next slot once it is free; then
// waits until the consumers have released every chunk. kv_issued counts the
// lane's chunks over the whole step (it keys the slots' mbarrier phases).
__device__ bool attn_stream(const ModelDesc& md, const StepDesc& sd, const Smem& sm, int layer,
                            const CUtensorMap* tmk, const CUtensorMap* tmv, uint32_t& kv_issued, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  const int ng = sd.attn_ng, spg = sd.attn_spg;
  const AttnBuf ab = attn_buf(sm);
  const AttnSlot SL = attn_slot_layout(md.dh, md.kv_q8);
  const int fa_i = md.layer[layer].fa_i;
  const int hkv = md.hkv;
  const int bw = SL.box_w / (md.kv_q8 ? 1 : 2);  // box width in elements
  const bool mine = lane < ng;
  int item = blockIdx.x, i = lane;
  AttnItem it{};
  bool done = !mine;
  auto seek = [&]() {
    while (!done) {
      if (item >= sd.n_attn_items) { done = true; break; }
      it = attn_item(sd, hkv, item);
      if (i < it.nch) break;
      item += gridDim.x;
      i = lane;
    }
  };
  seek();
  // the block's own item (at most one per block): all of its page ids at
  // once, so that issuing a page waits for no page-table round trip
  int* plist = reinterpret_cast<int*>(smem_raw + kOffRing + kRingBytes - kAttnPageListBytes);
  if (static_cast<int>(blockIdx.x) < sd.n_attn_items) {
    const AttnItem own = attn_item(sd, hkv, blockIdx.x);
    const int* src = md.page_table + static_cast<size_t>(sd.seq_id[own.si]) * md.max_pages_per_seq + own.cb;
    for (int c = lane; c < own.nch && c < kAttnPageList; c += 32) plist[c] = __ldcg(src + c);
  }
  __syncwarp();
  volatile int32_t* err = md.err;
  uint64_t t_idle = 0;
  bool ok = true;
  for (uint32_t sweep = 0;; ++sweep) {
    if (__all_sync(0xffffffffu, done)) break;
    bool issued = false;
    if (!done) {
      const int slot = lane * spg + static_cast<int>(kv_issued % static_cast<uint32_t>(spg));
      if (mbar_test(ab.empty + slot, ((kv_issued / spg) & 1u) ^ 1u)) {
        const int page = (item == static_cast<int>(blockIdx.x) && i < kAttnPageList)
                             ? plist[i]
                             : md.page_table[static_cast<size_t>(sd.seq_id[it.si]) * md.max_pages_per_seq + it.cb + i];
        const int row = ((fa_i * md.n_pages + page) * hkv + it.kh) * kChunk;
        uint8_t* dst = ab.slots + slot * SL.bytes;
        uint64_t* fb = ab.full + slot;
        mbar_arrive_expect_tx(fb, SL.tx_bytes);
        for (int bx = 0; bx < SL.nbox; ++bx) {
          tma_load_2d(dst + bx * kChunk * SL.box_w, tmk, bx * bw, row, fb, pol);
          tma_load_2d(dst + SL.v_off + bx * kChunk * SL.box_w, tmv, bx * bw, row, fb, pol);
        }
        if (md.kv_q8) {
          const int sb = kChunk * (md.dh / 32) * 2;
          bulk_g2s(dst + SL.ks_off, md.kv_ks + static_cast<size_t>(row) * (md.dh / 32), sb, fb, pol);
          bulk_g2s(dst + SL.vs_off, md.kv_vs + static_cast<size_t>(row) * (md.dh / 32), sb, fb, pol);
        }
        ++kv_issued;
        i += ng;
        seek();
        issued = true;
      }
    }
    if (__any_sync(0xffffffffu, issued)) {
      t_idle = 0;
    } else if ((sweep & 63u) == 63u) {
      if (*err != 0) { ok = false; break; }
      const uint64_t now = globaltimer();
      if (t_idle == 0) t_idle = now;
      else if (now - t_idle > sd.barrier_timeout_ns) { atomicCAS(md.err, 0, DEV_COPY_TIMEOUT); ok = false; break; }
    }
  }
  if (ok && mine && kv_issued > 0) {
    const uint32_t q = kv_issued - 1;
    ok = mbar_wait_bounded(ab.empty + lane * spg + q % spg, (q / spg) & 1u, md, sd.barrier_timeout_ns,
                           DEV_COPY_TIMEOUT);
  }
  return __all_sync(0xffffffffu, ok);
}

// The O^T accumulators of one warp: NQ n-tiles of 8 query rows each, MT
// m-tiles of 16 head dims (the warp's share of dh).
template <int NQ, int MT>
struct AttnAcc {
  float acc[NQ][MT][4];  // O^T: (dim rows g, g+8) x (columns 2c, 2c+1)
};

// 2^x by the MUFU instruction (ex2.approx.ftz: relative error near 2^-22,
// far below the binary16 rounding of P; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kAttnLazy = 8.f;

__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// One staged chunk of 16 tokens: the slot (or the step's own rows), the
// tokens that hold data, and the causal group (> 0: token t is masked for
// query row q when t > q / causal).
struct AttnSub {
  const uint8_t* cb;
  int nvalid, causal;
};

// A group's exchange area (attn_xslab bytes): score shares, P fragments,
// rescale factors and the final sums.
template <int NQ, int NU>
struct AttnX {
  float4* s;  // [wpg-1][NU][NQ][32]: the shares of the non-owners, in warp order
  uint2* p;   // [NQ][NU][32]: P^T fragments (binary16, transposed) of each chunk
  float2* f;  // [NQ][32]: rescale factors of columns 2c, 2c+1
  float2* l;  // [NQ][4]: final sums of columns 2c, 2c+1
  float4* m;  // [NQ][32]: the owner's running max and its lane's share of the sum
              // (m of columns 2c, 2c+1, then l of columns 2c, 2c+1)
  __device__ __forceinline__ AttnX(uint8_t* base, int wpg) {
    s = reinterpret_cast<float4*>(base);
    p = reinterpret_cast<uint2*>(base + (wpg - 1) * NU * NQ * 512);
    f = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(p) + NQ * NU * 256);
    l = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(f) + NQ * 256);
    m = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(l) + NQ * 32);
  }
};

// One step of warp dp of a group of wpg warps over NU chunks. The warp owns
// the 32-dim blocks j0 .. j0+JW-1 and forms their share of S^T = K Q^T for
// all NQ query n-tiles (rows past the item's own are zero and are not
// written out) and every chunk. The softmax of n-tile q is taken by warp
// q % wpg: it adds the shares (its own, then the others' in warp order),
// masks, takes the online-softmax step over the NU x 16 tokens and hands the
// group binary16 P^T fragments and the rescale factors; every warp then
// rescales its O^T and adds P V for the m-tiles of its blocks. bar_id is the
// group's named barrier (two per step). Slot layout (SL): K rows, V rows, q8
// block scales. Scores are in log2 units (Q carries log2(e) / sqrt(dh)).
// SWZ: 128-byte swizzled boxes (always for fp16; q8 when dh is a multiple of 128).
template <bool Q8, bool SWZ, int NQ, int JW, int NU>
__device__ __forceinline__ void attn_chunk(const AttnSub (&sub)[NU], const AttnSlot& SL, const __half* Qp,
                                           int qstride, int dh, int j0, int lane, int wpg, int dp,
                                           const AttnX<NQ, NU>& X, int bar_id, AttnAcc<NQ, 2 * JW>& st) {
  constexpr int BW = SWZ ? 128 : 64;  // bytes per box row
  constexpr int BB = kChunk * BW;     // bytes per box
  // with one chunk and one n-tile, the odd 32-dim blocks go to a second chain (latency)
  constexpr int NS = (NU == 1 && NQ == 1 && JW > 1) ? 2 : 1;
  const int g = lane >> 2, c = lane & 3;
  const int nblk = dh / 32;
  const int nthr = wpg * 32;
  float s[NU][NS][NQ][4];
#pragma unroll
  for (int u = 0; u < NU; ++u)
#pragma unroll
    for (int h = 0; h < NS; ++h)
#pragma unroll
      for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[u][h][q][e] = 0.f;
  const __half* qa = Qp + (lane & 7) * qstride + 8 * (lane >> 3);
#pragma unroll
  for (int jj = 0; jj < JW; ++jj) {
    const int j = j0 + jj;
    uint32_t b[NQ][4];
#pragma unroll
    for (int q = 0; q < NQ; ++q) ldsm_x4(b[q][0], b[q][1], b[q][2], b[q][3], qa + q * 8 * qstride + 32 * j);
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const uint8_t* kb = sub[u].cb;
      if (!Q8) {
        // lane c reads the 16-byte chunks 2c and 2c+1 of its box rows in turn
        const uint8_t* kr = kb + g * 128 + (((2 * c + (j & 1)) ^ g) << 4) + (j >> 1) * BB;
        const uint4 x = *reinterpret_cast<const uint4*>(kr);
        const uint4 y = *reinterpret_cast<const uint4*>(kr + 8 * 128);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float(&sj)[4] = s[u][jj % NS][q];
          mma16816(sj, x.x, y.x, x.y, y.y, b[q][0], b[q][1]);
          mma16816(sj, x.z, y.z, x.w, y.w, b[q][2], b[q][3]);
        }
      } else {
        const __half* ks = reinterpret_cast<const __half*>(kb + SL.ks_off);
        const int byte = 32 * j + 8 * c;
        int off;
        if (SWZ) {
          const int bb = byte & 127;
          off = (byte >> 7) * BB + g * 128 + ((((bb >> 4) ^ g) << 4) | (bb & 15));
        } else {
          off = g * 64 + byte;
        }
        const uint2 x = *reinterpret_cast<const uint2*>(kb + off);
        const uint2 y = *reinterpret_cast<const uint2*>(kb + off + 8 * BW);
        const uint32_t xx = x.x ^ 0x80808080u, xy = x.y ^ 0x80808080u;
        const uint32_t yx = y.x ^ 0x80808080u, yy = y.y ^ 0x80808080u;
        const uint32_t a0 = s8x2_to_h2(xx, 0x4140u), a1 = s8x2_to_h2(yx, 0x4140u);
        const uint32_t a2 = s8x2_to_h2(xx, 0x4342u), a3 = s8x2_to_h2(yx, 0x4342u);
        const uint32_t a4 = s8x2_to_h2(xy, 0x4140u), a5 = s8x2_to_h2(yy, 0x4140u);
        const uint32_t a6 = s8x2_to_h2(xy, 0x4342u), a7 = s8x2_to_h2(yy, 0x4342u);
        const float sg = __half2float(ks[g * nblk + j]), sg8 = __half2float(ks[(g + 8) * nblk + j]);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(t, a0, a1, a2, a3, b[q][0], b[q][1]);
          mma16816(t, a4, a5, a6, a7, b[q][2], b[q][3]);
          float(&sj)[4] = s[u][jj % NS][q];
          sj[0] = fmaf(sg, t[0], sj[0]);
          sj[1] = fmaf(sg, t[1], sj[1]);
          sj[2] = fmaf(sg8, t[2], sj[2]);
          sj[3] = fmaf(sg8, t[3], sj[3]);
        }
      }
    }
  }
  if (NS == 2) {
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[0][0][q][e] += s[0][NS - 1][q][e];
  }
  // shares to the owners (n-tile q is owned by warp q % wpg)
  int own = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (dp != own) {
      const int w = dp - (dp > own ? 1 : 0);
#pragma unroll
      for (int u = 0; u < NU; ++u)
        X.s[((w * NU + u) * NQ + q) * 32 + lane] =
            make_float4(s[u][0][q][0], s[u][0][q][1], s[u][0][q][2], s[u][0][q][3]);
    }
    own = own + 1 == wpg ? 0 : own + 1;
  }
  group_sync(bar_id, nthr);
  // the owner's softmax step for each of its n-tiles (one code body: the
  // tile's scores are first selected into sq)
  for (int q = dp; q < NQ; q += wpg) {
    float sq[NU][4];
#pragma unroll
    for (int u = 0; u < NU; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[u][0][0][e];
#pragma unroll
        for (int qq = 1; qq < NQ; ++qq) v = q == qq ? s[u][0][qq][e] : v;
        sq[u][e] = v;
      }
    for (int w = 0; w < wpg - 1; ++w) {
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const float4 v = X.s[((w * NU + u) * NQ + q) * 32 + lane];
        sq[u][0] += v.x;
        sq[u][1] += v.y;
        sq[u][2] += v.z;
        sq[u][3] += v.w;
      }
    }
    // masks: rows g / g+8 are tokens, columns q0 / q0+1 are query rows
    const int q0 = q * 8 + 2 * c;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int nv = sub[u].nvalid, cg = sub[u].causal;
      bool v0 = g < nv, v1 = v0, v2 = g + 8 < nv, v3 = v2;
      if (cg > 0) {
        v0 = v0 && g <= q0 / cg;
        v1 = v1 && g <= (q0 + 1) / cg;
        v2 = v2 && g + 8 <= q0 / cg;
        v3 = v3 && g + 8 <= (q0 + 1) / cg;
      }
      float(&sc)[4] = sq[u];
      sc[0] = v0 ? sc[0] : -INFINITY;
      sc[1] = v1 ? sc[1] : -INFINITY;
      sc[2] = v2 ? sc[2] : -INFINITY;
      sc[3] = v3 ? sc[3] : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[0], sc[2]));
      mx1 = fmaxf(mx1, fmaxf(sc[1], sc[3]));
    }
    // The reference m of a column moves only when a score passes it by more
    // than kAttnLazy (p then stays below 2^kAttnLazy): the common step needs
    // one vote instead of the max reduction, and no rescaling. The result is
    // the same softmax: O and l are both taken relative to m.
    float4 ml = X.m[q * 32 + lane];
    float mn0 = ml.x, mn1 = ml.y, a0 = 1.f, a1 = 1.f;
    if (__any_sync(0xffffffffu, mx0 > ml.x + kAttnLazy || mx1 > ml.y + kAttnLazy)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      mn0 = fmaxf(ml.x, mx0);
      mn1 = fmaxf(ml.y, mx1);
      a0 = ex2(ml.x - (mn0 == -INFINITY ? 0.f : mn0));
      a1 = ex2(ml.y - (mn1 == -INFINITY ? 0.f : mn1));
    }
    // a column with nothing visible yet keeps m = -inf and p = 0
    const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const float p0 = ex2(sq[u][0] - b0), p1 = ex2(sq[u][1] - b1);
      const float p2 = ex2(sq[u][2] - b0), p3 = ex2(sq[u][3] - b1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      X.p[(q * NU + u) * 32 + lane] = make_uint2(movm_trans(h2u(__floats2half2_rn(p0, p1))),
                                                 movm_trans(h2u(__floats2half2_rn(p2, p3))));
    }
    // l stays this lane's share (its tokens g, g+8); the lanes are added once, at the end
    ml = make_float4(mn0, mn1, fmaf(ml.z, a0, l0), fmaf(ml.w, a1, l1));
    X.m[q * 32 + lane] = ml;
    X.f[q * 32 + lane] = make_float2(a0, a1);
  }
  group_sync(bar_id, nthr);
  // every warp: rescale, then O^T += V^T P^T (A = V^T from the V rows by
  // ldmatrix.trans, B = the owners' P^T fragments)
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const float2 f = X.f[q * 32 + lane];
    if (!__any_sync(0xffffffffu, f.x != 1.f || f.y != 1.f)) continue;  // the max held: nothing to rescale
#pragma unroll
    for (int mi = 0; mi < 2 * JW; ++mi) {
      st.acc[q][mi][0] *= f.x;
      st.acc[q][mi][1] *= f.y;
      st.acc[q][mi][2] *= f.x;
      st.acc[q][mi][3] *= f.y;
    }
  }
  const int vt = (lane & 7) + 8 * (lane >> 4);  // token row this lane addresses
  const int vsub = (lane >> 3) & 1;
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    uint2 pb[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) pb[q] = X.p[(q * NU + u) * 32 + lane];
    const uint8_t* vrow = sub[u].cb + SL.v_off + vt * BW;
    const int nv = sub[u].nvalid;
    if (!Q8) {
      // tokens 2c, 2c+1 (a0, a1) and 2c+8, 2c+9 (a2, a3) beyond nvalid hold no data
      const uint32_t mlo = (2 * c < nv ? 0xffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
      const uint32_t mhi = (2 * c + 8 < nv ? 0xffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
      for (int mi = 0; mi < 2 * JW; ++mi) {
        const int M = 2 * j0 + mi;  // 16 dims = 32 bytes: box M / 4, chunks 2 (M % 4) + vsub
        const uint8_t* addr = vrow + (M >> 2) * BB + (((2 * (M & 3) + vsub) ^ (lane & 7)) << 4);
        uint32_t x0, x1, x2, x3;
        ldsm_x4_trans(x0, x1, x2, x3, addr);
        x0 &= mlo;
        x1 &= mlo;
        x2 &= mhi;
        x3 &= mhi;
#pragma unroll
        for (int q = 0; q < NQ; ++q) mma16816(st.acc[q][mi], x0, x1, x2, x3, pb[q].x, pb[q].y);
      }
    } else {
      // V = scale[token][block] x code, formed in binary16: the exact integer
      // code times the block scale of each of the lane's tokens 2c, 2c+1
      // (fragment registers 0, 1) and 2c+8, 2c+9 (registers 2, 3); tokens
      // beyond nvalid get scale 0
      const __half* vs = reinterpret_cast<const __half*>(sub[u].cb + SL.vs_off);
#pragma unroll
      for (int jb = 0; jb < JW; ++jb) {
        const int blk = j0 + jb;
        const __half z = __ushort_as_half(0);
        const __half2 s01 = __halves2half2(2 * c < nv ? vs[(2 * c) * nblk + blk] : z,
                                           2 * c + 1 < nv ? vs[(2 * c + 1) * nblk + blk] : z);
        const __half2 s89 = __halves2half2(2 * c + 8 < nv ? vs[(2 * c + 8) * nblk + blk] : z,
                                           2 * c + 9 < nv ? vs[(2 * c + 9) * nblk + blk] : z);
        const uint8_t* addr = SWZ ? vrow + (blk >> 2) * BB + (((2 * (blk & 3) + vsub) ^ (lane & 7)) << 4)
                                  : vrow + 32 * blk + 16 * vsub;
        uint32_t r0_, r1_, r2_, r3_;
        ldsm_x4_trans(r0_, r1_, r2_, r3_, addr);
        r0_ ^= 0x80808080u;
        r1_ ^= 0x80808080u;
        r2_ ^= 0x80808080u;
        r3_ ^= 0x80808080u;
        auto sc = [](uint32_t v, __half2 m) {
          const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&v), m);
          return h2u(h);
        };
        // m-rows g / g+8 of a tile are the block's even / odd dims
        const uint32_t e0 = sc(s8x2_to_h2(r0_, 0x4240u), s01), e1 = sc(s8x2_to_h2(r0_, 0x4341u), s01);
        const uint32_t e2 = sc(s8x2_to_h2(r2_, 0x4240u), s89), e3 = sc(s8x2_to_h2(r2_, 0x4341u), s89);
        const uint32_t o0 = sc(s8x2_to_h2(r1_, 0x4240u), s01), o1 = sc(s8x2_to_h2(r1_, 0x4341u), s01);
        const uint32_t o2 = sc(s8x2_to_h2(r3_, 0x4240u), s89), o3 = sc(s8x2_to_h2(r3_, 0x4341u), s89);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          mma16816(st.acc[q][2 * jb], e0, e1, e2, e3, pb[q].x, pb[q].y);
          mma16816(st.acc[q][2 * jb + 1], o0, o1, o2, o3, pb[q].x, pb[q].y);
        }
      }
    }
  }
}

// Head dim held by accumulator row `row` (0..15) of m-tile M.
template <bool Q8>
__device__ __forceinline__ int attn_dim(int M, int row) {
  if (!Q8) return M * 16 + row;
  return (M >> 1) * 32 + (M & 1) * 16 + (row < 8 ? 2 * row : 2 * (row - 8) + 1);
}

// binary16 nearest to amax / 127 (ties to even), in single precision only: a
// candidate from the single-precision quotient, then the midpoints to its
// neighbours compared exactly (127 x a midpoint of two binary16 values has at
// most 19 significant bits). amax >= 0.
__device__ __forceinline__ __half q8_block_scale(float amax) {
  const __half h = __float2half_rn(amax / 127.0f);
  const unsigned short u = __half_as_ushort(h);
  const float hf = __half2float(h);
  if (u < 0x7bffu) {  // the next binary16 up is finite
    const float up = __half2float(__ushort_as_half(static_cast<unsigned short>(u + 1)));
    const float pm = 127.0f * (0.5f * (hf + up));
    if (amax > pm || (amax == pm && (u & 1u))) return __ushort_as_half(static_cast<unsigned short>(u + 1));
  }
  if (u > 0 && u < 0x7c00u) {
    const float dn = __half2float(__ushort_as_half(static_cast<unsigned short>(u - 1)));
    const float pm = 127.0f * (0.5f * (dn + hf));
    if (amax < pm || (amax == pm && (u & 1u))) return __ushort_as_half(static_cast<unsigned short>(u - 1));
  }
  return h;
}

// round-half-even of val / d, clamped to [-127, 127] (0 when d = 0), exactly:
// the single-precision quotient rounded, then corrected by the exact remainder
// val - q d (q d has at most 18 significant bits)
__device__ __forceinline__ int q8_code(float val, float d) {
  if (d == 0.f) return 0;
  float q = rintf(val / d);
  const float r = fmaf(-q, d, val), h = 0.5f * d;
  const bool odd = (static_cast<int>(q) & 1) != 0;
  if (r > h || (r == h && odd)) q += 1.f;
  else if (r < -h || (r == -h && odd)) q -= 1.f;
  return static_cast<int>(fminf(fmaxf(q, -127.f), 127.f));
}

// K (with RoPE) and V of the step's own row t for kv head kh, from the input
// projection's output (kr, vr; rope: the row's (cos, sin) per pair), rounded
// (fp16 pool) or quantised (q8 pool: per 32-dim block, scale = binary16 of
// amax / 127, code = round(x / scale)) into the pool at (page, slot) and, as
// stored, into row t of the new-rows chunk. Lane l holds the dims l + 32 j of
// each half of the row: RoPE pairs dim d < dh/2 with d + dh/2 in the same lane.
__device__ __noinline__ void attn_new_row(const ModelDesc& md, const float* kr, const float* vr, const float2* rope,
                                          int fa_i, int page, int kh, int slot, uint8_t* newt, const AttnSlot& SL,
                                          int t, int lane) {
  constexpr int kH = kMaxDh / 64;  // 32-dim blocks per half row, at most
  const int dh = md.dh, nh = dh / 64;
  const bool q8 = md.kv_q8 != 0;
  const size_t row = ((static_cast<size_t>(fa_i) * md.n_pages + page) * md.hkv + kh) * md.page_tokens + slot;
#pragma unroll 1
  for (int w = 0; w < 2; ++w) {
    float x[2 * kH];  // [half * kH + j]
#pragma unroll
    for (int j = 0; j < kH; ++j)
      if (j < nh) {
        const int d = 32 * j + lane;
        if (w == 0) {
          const float a = __ldcg(kr + d), b = __ldcg(kr + d + dh / 2);
          const float2 cs = __ldcg(rope + d);
          x[j] = a * cs.x - b * cs.y;
          x[kH + j] = a * cs.y + b * cs.x;
        } else {
          x[j] = __ldcg(vr + d);
          x[kH + j] = __ldcg(vr + d + dh / 2);
        }
      }
    uint8_t* tile = newt + (w ? SL.v_off : 0);
    void* pool = w ? md.kv_v : md.kv_k;
    if (!q8) {
      __half* dst = reinterpret_cast<__half*>(pool) + row * dh;
#pragma unroll
      for (int i = 0; i < 2 * kH; ++i) {
        const int hf = i / kH, j = i % kH;
        if (j < nh) {
          const int d = 32 * (hf * nh + j) + lane;
          const __half hv = __float2half_rn(x[i]);
          dst[d] = hv;
          *reinterpret_cast<__half*>(tile + kv_off(SL, t, 2 * d)) = hv;
        }
      }
    } else {
      int8_t* codes = reinterpret_cast<int8_t*>(pool) + row * dh;
      uint16_t* scales = (w ? md.kv_vs : md.kv_ks) + row * (dh / 32);
      __half* tscale = reinterpret_cast<__half*>(newt + (w ? SL.vs_off : SL.ks_off)) + t * (dh / 32);
#pragma unroll
      for (int i = 0; i < 2 * kH; ++i) {
        const int hf = i / kH, j = i % kH;
        if (j < nh) {
          const int blk = hf * nh + j, d = 32 * blk + lane;
          const __half d16 = q8_block_scale(warp_max(fabsf(x[i])));
          const int q = q8_code(x[i], __half2float(d16));
          codes[d] = static_cast<int8_t>(q);
          tile[kv_off(SL, t, d)] = static_cast<uint8_t>(static_cast<int8_t>(q));
          if (lane == 0) {
            scales[blk] = __half_as_ushort(d16);
            tscale[blk] = d16;
          }
        }
      }
    }
  }
}

// Test hook: the q8 block codec of attn_new_row on n_blocks blocks of 32
// floats, one warp per block (codes q[32 b + i], scales d16[b]).
__global__ void q8_encode_kernel(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d16) {
  const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (b >= n_blocks) return;  // whole warps: blockDim is a multiple of 32
  const float v = x[b * 32 + lane];
  const __half h = q8_block_scale(warp_max(fabsf(v)));
  q[b * 32 + lane] = static_cast<int8_t>(q8_code(v, __half2float(h)));
  if (lane == 0) d16[b] = __half_as_ushort(h);
}

cudaError_t launch_q8_encode(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d16, cudaStream_t stream) {
  constexpr int kBlock = 256;
  const int64_t grid = (n_blocks * 32 + kBlock - 1) / kBlock;
  if (n_blocks <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  q8_encode_kernel<<<static_cast<unsigned>(grid), kBlock, 0, stream>>>(x, n_blocks, q, d16);
  return cudaGetLastError();
}

// One row of K or V that an earlier phase of this launch stored into the pool
// (an MTP draft pass reads back the positions of the catch-up rows and of the
// passes before it), copied as stored into row t of the new-rows chunk.
__device__ void attn_load_kv(const ModelDesc& md, int fa_i, int page, int kh, int slot, int which, uint8_t* tile,
                             __half* tile_scales, const AttnSlot& SL, int t, int lane) {
  const int dh = md.dh;
  const size_t row = ((static_cast<size_t>(fa_i) * md.n_pages + page) * md.hkv + kh) * md.page_tokens + slot;
  if (!md.kv_q8) {
    const unsigned short* src = reinterpret_cast<const unsigned short*>(which ? md.kv_v : md.kv_k) + row * dh;
    for (int d = lane; d < dh; d += 32)
      *reinterpret_cast<unsigned short*>(tile + kv_off(SL, t, 2 * d)) = __ldcg(src + d);
  } else {
    const signed char* codes = reinterpret_cast<const signed char*>(which ? md.kv_v : md.kv_k) + row * dh;
    const unsigned short* scales = (which ? md.kv_vs : md.kv_ks) + row * (dh / 32);
    for (int d = lane; d < dh; d += 32)
      tile[kv_off(SL, t, d)] = static_cast<uint8_t>(__ldcg(codes + d));
    for (int b = lane; b < dh / 32; b += 32)
      tile_scales[t * (dh / 32) + b] = __ushort_as_half(__ldcg(scales + b));
  }
}

static_assert(attn_qbytes(kMaxQRows / 8, kMaxDh) + 16384 + 16 <= kPhaseBytes, "attention shared memory");
// the merge's weights (2 x rows x partials + rows floats) stay below the
// phase's flag word: the host keeps rows x partials within kAttnCombineFloats
static_assert(kAttnBarOff + 2 * kAttnMaxSlots * 8 <= kMiscBytes, "attention mbarriers");

// Every block of a (sequence, kv head) merges its share of the partials
// (one per warp group of every split block) once all of them are written:
// split block j takes the output float4s j, j + nblocks, ... of the head's
// [qrows][dh/4] output. First every partial's (m, l) of every row goes to
// shared memory in one batch of loads; then per row the weights 2^(m_s - M)
// and 1/sum(l_s w_s); then groups of 4 threads sum one output float4 over the
// partials (each thread a quarter of them, all its loads in flight) and a
// shuffle adds the four.
__device__ __noinline__ void attn_combine(const ModelDesc& md, const StepDesc& sd, int si, int kh, int nblocks,
                                          int ngroups, int qrows, int row0, int j, float* wsm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int dh = md.dh, grp = md.hq / md.hkv;
  const int item0 = sd.seq_item0[si] + kh * nblocks;
  const int nsplit = nblocks * ngroups;  // partials: every group of every split block
  const int n = qrows * nsplit;
  float* wm = wsm;          // [qrows][nsplit]: m, then the weight
  float* wl = wsm + n;      // [qrows][nsplit]: l
  float* inv = wsm + 2 * n;  // [qrows]
  auto part = [&](int sp, int r) {
    return md.attn_part +
           ((static_cast<size_t>(item0 + sp / ngroups) * kMaxAttnGroups + sp % ngroups) * md.part_rows + r) *
               md.part_stride;
  };
  for (int base = 0; base < n; base += kThreads * 8) {
    float2 ml[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int idx = base + b * kThreads + tid;
      ml[b] = idx < n ? __ldcg(reinterpret_cast<const float2*>(part(idx % nsplit, idx / nsplit) + dh))
                      : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int idx = base + b * kThreads + tid;
      if (idx < n) {
        wm[idx] = ml[b].x;
        wl[idx] = ml[b].y;
      }
    }
  }
  math_sync();
  for (int r = warp; r < qrows; r += kWarps) {
    float mloc = -INFINITY;
    for (int sp = lane; sp < nsplit; sp += 32) mloc = fmaxf(mloc, wm[r * nsplit + sp]);
    const float M = warp_max(mloc);
    float lloc = 0.f;
    for (int sp = lane; sp < nsplit; sp += 32) {
      const float ms = wm[r * nsplit + sp];
      const float w = ms == -INFINITY ? 0.f : exp2f(ms - M);
      wm[r * nsplit + sp] = w;
      lloc = fmaf(wl[r * nsplit + sp], w, lloc);
    }
    const float tot = warp_sum(lloc);
    if (lane == 0) inv[r] = 1.0f / tot;
  }
  math_sync();
  const int d4n = dh / 4, total = qrows * d4n;
  constexpr int kG = 4;                     // threads per output float4
  constexpr int kSlots = kThreads / kG;     // outputs per pass of the block
  const int q = tid & (kG - 1), slot = tid / kG;
  // the pass loop is warp-uniform (the shuffles below need the whole warp)
  for (int pass = 0; j + nblocks * (warp * (32 / kG) + kSlots * pass) < total; ++pass) {
    const int o = j + nblocks * (slot + kSlots * pass);
    const bool valid = o < total;
    const int r = valid ? o / d4n : 0, d4 = valid ? o - r * d4n : 0;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = q; sp0 < nsplit; sp0 += kG * 16) {
      float4 v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int sp = sp0 + kG * u;
        v[u] = (valid && sp < nsplit) ? __ldcg(reinterpret_cast<const float4*>(part(sp, r)) + d4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int sp = sp0 + kG * u;
        const float w = (valid && sp < nsplit) ? wm[r * nsplit + sp] : 0.f;
        a.x = fmaf(w, v[u].x, a.x);
        a.y = fmaf(w, v[u].y, a.y);
        a.z = fmaf(w, v[u].z, a.z);
        a.w = fmaf(w, v[u].w, a.w);
      }
    }
#pragma unroll
    for (int off = 1; off < kG; off <<= 1) {
      a.x += __shfl_xor_sync(0xffffffffu, a.x, off);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, off);
      a.z += __shfl_xor_sync(0xffffffffu, a.z, off);
      a.w += __shfl_xor_sync(0xffffffffu, a.w, off);
    }
    if (valid && q == 0) {
      const float iv = inv[r];
      const int t = r / grp, hh = kh * grp + r % grp;
      float4* op = reinterpret_cast<float4*>(md.o + static_cast<size_t>(row0 + t) * md.o_stride + hh * dh) + d4;
      *op = make_float4(a.x * iv, a.y * iv, a.z * iv, a.w * iv);
    }
  }
}

// Bounded wait until every split of (sequence, kv head) `key` has announced
// its partial for attention phase number `ord` of this launch: the counter
// only grows within a launch (the host clears it before each), so the phase's
// target is (ord + 1) x nsplit. False (and the error word set) on timeout or
// when another block has already reported an error.
__device__ bool attn_splits_ready(const ModelDesc& md, const StepDesc& sd, int key, int ord, int nsplit) {
  const uint32_t target = static_cast<uint32_t>(ord + 1) * static_cast<uint32_t>(nsplit);
  volatile int32_t* err = md.err;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(md.attn_tickets + key) >= target) return true;
    if ((it & 31u) == 31u) {
      if (*err != 0) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > sd.barrier_timeout_ns || it > (1u << 30)) {
        atomicCAS(md.err, 0, DEV_BARRIER_TIMEOUT);
        return false;
      }
    }
  }
}

// mp > 0: MTP draft pass mp. Only the first row of each sequence is real: it
// sits at slot k = mtp_row[si].slot (position = cached length + k) with RoPE
// angles from mtp_rope; the new-rows chunk holds the slots 0..k-1 that earlier
// phases of this launch stored (read back) and the row's own K/V at slot k,
// all visible to it.
template <bool Q8, bool SWZ, int NQ, int JW>
__device__ __noinline__ bool attn_phase(const ModelDesc& md, const StepDesc& sd, int layer, const Smem& sm,
                                        WarpCtx& wc, int mp) {
  const LayerDesc& L = md.layer[layer];
  const int fa_i = L.fa_i;
  const int dh = md.dh, hkv = md.hkv, grp = md.hq / md.hkv;
  const int tid = threadIdx.x, warp = wc.warp, lane = wc.lane;
  const int g = lane >> 2, c = lane & 3;
  const AttnSlot SL = attn_slot_layout(dh, Q8 ? 1 : 0);
  const AttnBuf ab = attn_buf(sm);
  // a group of wpg warps takes one chunk at a time; each of its warps owns
  // every query n-tile and the dims of JW 32-dim blocks
  const int ng = sd.attn_ng, wpg = sd.attn_wpg, spg = sd.attn_spg;
  const int tg = warp / wpg, dp = warp % wpg;
  const bool in_group = tg < ng;
  const int j0 = dp * JW;
  const int nmt = 2 * JW, mt0 = 2 * j0;
  const int qstride = dh + 8;
  __half* Qp = reinterpret_cast<__half*>(sm.phase());
  uint8_t* newt = sm.phase() + attn_qbytes(NQ, dh);
  // this group's exchange area
  constexpr int NU = attn_nu(NQ, Q8 ? 1 : 0);
  const AttnX<NQ, NU> X(sm.phase() + attn_xoff(NQ, dh, Q8 ? 1 : 0) + tg * attn_xslab(wpg, NQ, Q8 ? 1 : 0), wpg);
  int* flag = reinterpret_cast<int*>(sm.phase() + kPhaseBytes - 16);
  const float q_scale = 1.4426950408889634f / sqrtf(static_cast<float>(dh));  // log2(e) / sqrt(dh)
  const int kq_off = 2 * md.hq * dh;    // k after q and gate
  const int vq_off = kq_off + hkv * dh;  // v after k
  bool ok = true;

  for (int item = blockIdx.x; item < sd.n_attn_items; item += gridDim.x) {
    const AttnItem it = attn_item(sd, hkv, item);
    const int si = it.si, kh = it.kh;
    const int seq = sd.seq_id[si], T = sd.seq_T[si], row0 = sd.seq_row0[si], Lc = sd.seq_len[si];
    const int qrows = T * grp, nq = (qrows + 7) / 8;
    const bool last = it.j == it.nsplit - 1;
    const int* pt = md.page_table + static_cast<size_t>(seq) * md.max_pages_per_seq;

    // Q (RoPE, 1/sqrt(dh), binary16), head dims in the order the K fragments
    // present them; rows past qrows are zero
    // batches of 4 pairs per thread: all of a batch's loads are issued before
    // its shared-memory stores
    const int nqe = NQ * 8 * (dh / 2);  // every n-tile of the variant: rows past qrows are zero
    for (int base = 0; base < nqe; base += kThreads * 4) {
      float qa[4][2], qb[4][2];
      float2 qc[4][2];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int idx = base + bb * kThreads + tid;
        const int qr = idx / (dh / 2), pp = 2 * (idx % (dh / 2));
        const int sidx = pp >> 4, l16 = pp & 15, j = sidx >> 1, h = sidx & 1, cc = (l16 & 7) >> 1, hi = l16 >> 3;
        const int d = Q8 ? 32 * j + 8 * cc + 4 * h + 2 * hi : 64 * (j >> 1) + 16 * cc + 8 * (j & 1) + 4 * h + 2 * hi;
        const bool in = idx < nqe && qr < qrows;
        const int t = in ? qr / grp : 0, hh = kh * grp + (in ? qr % grp : 0), row = row0 + t;
        const float* q = md.yin + static_cast<size_t>(row) * md.n_in_max + hh * dh;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = (d + e) % (dh / 2);
          qa[bb][e] = in ? __ldcg(q + i) : 0.f;
          qb[bb][e] = in ? __ldcg(q + i + dh / 2) : 0.f;
          qc[bb][e] = !in ? make_float2(0.f, 0.f)
                          : mp ? __ldcg(md.mtp_rope + si * (kMaxDh / 2) + i) : sd.rope[row][i];
        }
      }
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int idx = base + bb * kThreads + tid;
        if (idx < nqe) {
          const int qr = idx / (dh / 2), pp = 2 * (idx % (dh / 2));
          const int sidx = pp >> 4, l16 = pp & 15, j = sidx >> 1, h = sidx & 1, cc = (l16 & 7) >> 1, hi = l16 >> 3;
          const int d = Q8 ? 32 * j + 8 * cc + 4 * h + 2 * hi : 64 * (j >> 1) + 16 * cc + 8 * (j & 1) + 4 * h + 2 * hi;
          float v[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float a = qa[bb][e], b = qb[bb][e];
            const float2 cs = qc[bb][e];
            v[e] = (d + e < dh / 2 ? a * cs.x - b * cs.y : a * cs.y + b * cs.x) * q_scale;
          }
          *reinterpret_cast<__half2*>(Qp + qr * qstride + pp) = __floats2half2_rn(v[0], v[1]);
        }
      }
    }
    // the step's own rows (last split): RoPE k, store K/V into the pool, and
    // keep the stored values as one more chunk, causal over the T rows (a
    // draft pass: the earlier slots read back plus its own row, all visible)
    const int k_own = mp ? min(max(__ldcg(md.mtp_row + 2 * si + 1), 0), kChunk - 1) : 0;
    const int n_new = mp ? k_own + 1 : T;
    if (last) {
      for (int idx = tid; idx < SL.tx_bytes / 16; idx += kThreads)
        reinterpret_cast<uint4*>(newt)[idx] = make_uint4(0u, 0u, 0u, 0u);
      math_sync();
      for (int t = warp; t < n_new; t += kWarps) {
        const int pos = Lc + t;
        const int page = pt[pos / md.page_tokens], slot = pos % md.page_tokens;
        if (mp && t < k_own) {
          attn_load_kv(md, fa_i, page, kh, slot, 0, newt, reinterpret_cast<__half*>(newt + SL.ks_off), SL, t, lane);
          attn_load_kv(md, fa_i, page, kh, slot, 1, newt + SL.v_off, reinterpret_cast<__half*>(newt + SL.vs_off), SL,
                       t, lane);
          continue;
        }
        const int row = row0 + (mp ? 0 : t);
        const float* kr = md.yin + static_cast<size_t>(row) * md.n_in_max + kq_off + kh * dh;
        const float* vr = md.yin + static_cast<size_t>(row) * md.n_in_max + vq_off + kh * dh;
        const float2* rope = mp ? md.mtp_rope + si * (kMaxDh / 2) : sd.rope[row];
        attn_new_row(md, kr, vr, rope, fa_i, page, kh, slot, newt, SL, t, lane);
      }
    }
    math_sync();

    AttnAcc<NQ, 2 * JW> st;
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (in_group && q % wpg == dp) X.m[q * 32 + lane] = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
#pragma unroll
      for (int mi = 0; mi < 2 * JW; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.acc[q][mi][e] = 0.f;
    }
    // this block's chunks round-robin over the groups; the step's own rows
    // (last split) are one more chunk, read from the new-rows tile. Every warp
    // of a group runs every chunk (also after a failed wait: its result is
    // then void) so that the group's barriers always meet.
    if (in_group) {
      const int nv = it.nch + (last ? 1 : 0);
      for (int i = tg; i < nv; i += NU * ng) {
        // chunks i, i + ng, ... (NU of them, those past nv void): cached pages
        // come from the group's slots in order, the step's own rows from newt
        AttnSub sub[NU];
        int slot[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int iu = i + u * ng;
          slot[u] = -1;
          sub[u] = AttnSub{newt, 0, 0};
          if (iu < it.nch) {
            const uint32_t pos = wc.kv_pos + u;
            slot[u] = tg * spg + static_cast<int>(pos % static_cast<uint32_t>(spg));
            if (ok)
              ok = mbar_wait_bounded(ab.full + slot[u], (pos / spg) & 1u, md, sd.barrier_timeout_ns,
                                     DEV_COPY_TIMEOUT);
            sub[u] = AttnSub{ab.slots + slot[u] * SL.bytes, min(kChunk, Lc - (it.cb + iu) * kChunk), 0};
          } else if (iu < nv) {
            sub[u] = AttnSub{newt, n_new, mp ? 0 : grp};
          }
        }
        attn_chunk<Q8, SWZ, NQ, JW, NU>(sub, SL, Qp, qstride, dh, j0, lane, wpg, dp, X, 2 + tg, st);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < NU; ++u)
          if (slot[u] >= 0) {
            if (lane == 0) mbar_arrive(ab.empty + slot[u]);
            ++wc.kv_pos;
          }
      }
    }

    // write out: directly if this block's one group holds the whole head,
    // else this group's partial (unnormalised O, m, l) for the merge
    const bool merged = it.nsplit > 1 || ng > 1;
    float* part = md.attn_part + (static_cast<size_t>(item) * kMaxAttnGroups + tg) * md.part_rows * md.part_stride;
    if (in_group) {
      // the owners' sums (lanes added) for every warp of the group; the owners
      // also write m and l of a partial
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q % wpg == dp) {
          const float4 ml = X.m[q * 32 + lane];
          float lq[2] = {ml.z, ml.w};
          const float mq[2] = {ml.x, ml.y};
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) lq[e] += __shfl_xor_sync(0xffffffffu, lq[e], o);
          if (g == 0) X.l[q * 4 + c] = make_float2(lq[0], lq[1]);
          if (merged && g == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int qr = q * 8 + 2 * c + e;
              if (qr < qrows) {
                __stcg(part + static_cast<size_t>(qr) * md.part_stride + dh, mq[e]);
                __stcg(part + static_cast<size_t>(qr) * md.part_stride + dh + 1, lq[e]);
              }
            }
          }
        }
      }
      group_sync(2 + tg, wpg * 32);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q < nq) {
          const float2 lq = X.l[q * 4 + c];
          // this lane's two query columns of n-tile q: destination row and scale
          float* dst[2];
          float sc[2];
          bool okq[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int qr = q * 8 + 2 * c + e;
            okq[e] = qr < qrows;
            const int t = qr / grp, hh = kh * grp + qr % grp;
            dst[e] = !merged ? md.o + static_cast<size_t>(row0 + t) * md.o_stride + hh * dh
                             : part + static_cast<size_t>(qr) * md.part_stride;
            sc[e] = !merged ? 1.0f / (e ? lq.y : lq.x) : 1.0f;
          }
#pragma unroll
          for (int mi = 0; mi < 2 * JW; ++mi)
            if (mi < nmt)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (okq[e & 1])
                  __stcg(dst[e & 1] + attn_dim<Q8>(mt0 + mi, e < 2 ? g : g + 8), st.acc[q][mi][e] * sc[e & 1]);
        }
      }
    }
    if (merged) {
      // announce this block's partials, wait for the others, merge this block's share
      __threadfence();
      math_sync();
      if (tid == 0) {
        const int key = si * hkv + kh;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(md.attn_tickets + key) : "memory");
        *flag = attn_splits_ready(md, sd, key, fa_i + mp, it.nsplit) ? 1 : 0;
      }
      math_sync();
      if (*flag) attn_combine(md, sd, si, kh, it.nsplit, ng, qrows, row0, it.j, reinterpret_cast<float*>(sm.phase()));
      else ok = false;
    }
    math_sync();
  }
  return ok;
}

// The attention variant for the step's query n-tiles per (sequence, kv head)
// and 32-dim blocks per warp: each warp holds nq n-tiles x 2 jw m-tiles of O^T.
template <bool Q8, bool SWZ>
__device__ __forceinline__ bool attn_dispatch(int nq, int jw, const ModelDesc& md, const StepDesc& sd, int layer,
                                              const Smem& sm, WarpCtx& wc, int mp) {
  switch (nq) {
    case 1:
      if (jw == 4) return attn_phase<Q8, SWZ, 1, 4>(md, sd, layer, sm, wc, mp);
      return attn_phase<Q8, SWZ, 1, 2>(md, sd, layer, sm, wc, mp);
    case 2: return attn_phase<Q8, SWZ, 2, 2>(md, sd, layer, sm, wc, mp);
    case 3: return attn_phase<Q8, SWZ, 3, 2>(md, sd, layer, sm, wc, mp);
    case 4: return attn_phase<Q8, SWZ, 4, 1>(md, sd, layer, sm, wc, mp);
    case 5: return attn_phase<Q8, SWZ, 5, 1>(md, sd, layer, sm, wc, mp);
    default: return attn_phase<Q8, SWZ, 6, 1>(md, sd, layer, sm, wc, mp);
  }
}

static_assert(kWarps * (2 * kMaxT * 128 + kMaxT * 10) * 4 <= kPhaseBytes, "Gated DeltaNet shared memory");

// ------------------------------------------------------------ lm argmax
// When lm_head's reduction is sliced, every tile is split and its logits were
// summed in md.logits; after the barrier each warp scans tiles gid, gid +
// (warps), ... and merges them into its top-1 record (ties: lowest index).
__device__ __noinline__ void lm_argmax(const ModelDesc& md, const StepDesc& sd, const GemmDesc& g,
                                      const WarpCtx& wc) {
  const int R = sd.R, lane = wc.lane;
  const int nw = gridDim.x * kWarps;
  const int ntile = g.n_tiles;
  float b[kMaxRows];
  int bi[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    b[r] = -FLT_MAX;
    bi[r] = 0x7fffffff;
  }
  for (int t = wc.gid; t < ntile; t += nw) {
    const int n = t * kTileRows + lane;
    if (n < g.n_out) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
        if (r < R) {
          const float x = __ldcg(md.logits + static_cast<size_t>(r) * md.V + n);
          if (!isfinite(x)) atomicOr(&md.err[1], 1);
          if (md.dbg_logits && g.dump) md.dbg_logits[static_cast<size_t>(r) * md.V + n] = x;
          top1_merge(b[r], bi[r], x, n);
        }
    }
  }
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r)
    if (r < R) {
      float x = b[r];
      int ix = bi[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ox = __shfl_xor_sync(0xffffffffu, x, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
        top1_merge(x, ix, ox, oi);
      }
      if (lane == 0) {
        const size_t at = static_cast<size_t>(wc.gid) * kMaxRows + r;
        float rb = md.top_val[at];
        int ri = md.top_idx[at];
        top1_merge(rb, ri, x, ix);
        md.top_val[at] = rb;
        md.top_idx[at] = ri;
      }
    }
}

// ------------------------------------------------------------------ verify
// Block 0: argmax of every row over all warps' top-2 records (lowest index on
// exact ties), then per sequence the longest prefix of drafts that equal the
// previous row's argmax; emitted = accepted drafts + the bonus argmax. A
// sequence of prompt rows emits nothing, or the argmax of its last row when
// the rows end its prompt.
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
      if (sd.seq_prompt[si]) {  // prompt rows: no verification; one token when the prompt ends
        const int emits = sd.seq_prompt[si] == 2 ? 1 : 0;
        if (emits) md.out[kOutTokens + at++] = am[row0 + T - 1];
        md.out[kOutCounts + si] = emits;
        continue;
      }
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

// ------------------------------------------------------- MTP draft head
// One element of the embedding matrix (Q4 super-blocks, row `tok`).
__device__ __forceinline__ float embed_value(const ModelDesc& md, int tok, int k) {
  const int nsbH = md.H / 256, sb = k >> 8, j = (k & 255) >> 5, i = k & 31;
  const uint8_t* blk = md.embed + (static_cast<size_t>(tok) * nsbH + sb) * 144;
  const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
  const uint64_t lo64 = hdr.y | (static_cast<uint64_t>(hdr.z) << 32);
  const uint64_t mid64 = hdr.z | (static_cast<uint64_t>(hdr.w) << 32);
  const float sc = static_cast<float>((lo64 >> (6 * j)) & 63u);
  const float m = static_cast<float>((mid64 >> (16 + 6 * j)) & 63u);
  const uint8_t byte = __ldg(blk + 16 + 16 * j + (i % 16));
  const int q = i < 16 ? (byte & 15) : (byte >> 4);
  return (d * sc) * static_cast<float>(q) - dmin * m;
}

// Input rows of MTP draft pass p, one block per step row r:
//   mtp_in[r] = [RMSNorm(h) w_h ; RMSNorm(embed(tok)) w_e]
// with (h, tok) = (final hidden state of row r, its greedy token) in pass 0 and
// (the previous pass's hidden output, its draft) for the first row of each
// sequence in later passes (the other rows are zero). Also clears x[r], which
// W_fc's epilogue adds into, and the draft-logit rows the sliced lm_head sums into.
__device__ __noinline__ void mtp_input_phase(const ModelDesc& md, const StepDesc& sd, int p, const Smem& sm) {
  const int H = md.H, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    const int stride = gridDim.x * kThreads, t0 = blockIdx.x * kThreads + tid;
    for (int idx = t0; idx < sd.R * md.draft_vocab; idx += stride)
      md.logits[static_cast<size_t>(idx / md.draft_vocab) * md.V + idx % md.draft_vocab] = 0.f;
  }
  float* red = sm.misc() + 512;  // [warp][2] partial sums of squares
  for (int r = blockIdx.x; r < sd.R; r += gridDim.x) {
    const int si = sd.row_si[r];
    const bool real = p == 0 || r == sd.seq_row0[si];
    const float* h = p == 0 ? md.x + static_cast<size_t>(r) * H : md.mtp_h + static_cast<size_t>(si) * H;
    // (an all-NaN row leaves no argmax: the non-finite flag reports it; keep the index in range)
    const int tok = !real ? 0 : min(max(p == 0 ? __ldcg(md.out + kOutArgmax + r) : __ldcg(md.mtp_row + 2 * si), 0),
                                    md.V - 1);
    float* dst = md.mtp_in + static_cast<size_t>(r) * 2 * H;
    float sh = 0.f, se = 0.f;
    for (int k = tid; k < H; k += kThreads) {
      const float hv = real ? __ldcg(h + k) : 0.f;
      const float ev = real ? embed_value(md, tok, k) : 0.f;
      sh = fmaf(hv, hv, sh);
      se = fmaf(ev, ev, se);
      dst[k] = hv;
      dst[H + k] = ev;
    }
    sh = warp_sum(sh);
    se = warp_sum(se);
    if (lane == 0) {
      red[2 * warp] = sh;
      red[2 * warp + 1] = se;
    }
    math_sync();
    float th = 0.f, te = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      th += red[2 * w];
      te += red[2 * w + 1];
    }
    const float rh = 1.0f / sqrtf(th / static_cast<float>(H) + md.eps);
    const float re = 1.0f / sqrtf(te / static_cast<float>(H) + md.eps);
    for (int k = tid; k < H; k += kThreads) {
      dst[k] = dst[k] * rh * md.mtp_norm_h[k];
      dst[H + k] = dst[H + k] * re * md.mtp_norm_e[k];
      md.x[static_cast<size_t>(r) * H + k] = 0.f;
    }
    math_sync();  // red is reused by the next row
  }
}

// Block 0: draft p of every sequence = argmax over the draft vocabulary of
// its source row (pass 0: the last accepted row a; later passes: the first
// row), lowest index on ties. Unless p is the last pass, it also prepares
// pass p+1: the token (this draft), the slot a + p + 1, its RoPE angles in
// double precision, and the hidden state (the source row's x).
__device__ __noinline__ void draft_phase(const ModelDesc& md, const StepDesc& sd, int p) {
  if (blockIdx.x != 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nrec = gridDim.x * kWarps;
  for (int si = warp; si < sd.n_seq; si += kWarps) {
    const int a = __ldcg(md.out + kOutCounts + si) - 1;
    const int rs = p == 0 ? sd.seq_row0[si] + a : sd.seq_row0[si];
    float b1 = -FLT_MAX;
    int i1 = 0x7fffffff;
    for (int gidx = lane; gidx < nrec; gidx += 32)
      top1_merge(b1, i1, __ldcg(md.top_val + static_cast<size_t>(gidx) * kMaxRows + rs),
                 __ldcg(md.top_idx + static_cast<size_t>(gidx) * kMaxRows + rs));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob1 = __shfl_xor_sync(0xffffffffu, b1, o);
      const int oi1 = __shfl_xor_sync(0xffffffffu, i1, o);
      top1_merge(b1, i1, ob1, oi1);
    }
    if (lane == 0) md.out[kOutDrafts + si * kMaxDraft + p] = i1;
    if (p + 1 < md.n_draft) {
      const int k = a + p + 1;
      if (lane == 0) {
        md.mtp_row[2 * si] = i1;
        md.mtp_row[2 * si + 1] = k;
      }
      const double pos = static_cast<double>(sd.seq_len[si] + k);
      for (int i = lane; i < md.dh / 2; i += 32) {
        double sn, cs;
        sincos(pos * md.inv_freq[i], &sn, &cs);
        md.mtp_rope[si * (kMaxDh / 2) + i] = make_float2(static_cast<float>(cs), static_cast<float>(sn));
      }
      for (int k2 = lane; k2 < md.H; k2 += 32)
        md.mtp_h[static_cast<size_t>(si) * md.H + k2] = __ldcg(md.x + static_cast<size_t>(rs) * md.H + k2);
    }
  }
}

// ------------------------------------------------------------ the producer
#ifndef MK_PRODUCER_NAP
#define MK_PRODUCER_NAP 0
#endif
constexpr unsigned kProducerNapNs = MK_PRODUCER_NAP;  // producer back-off when every ring is full (ns)

// Lanes 0..kWarps-1 each walk one math warp's unit sequence; the warp stays
// converged: every sweep, each lane issues its next unit if that unit's slot
// has been released, then the sweep repeats until every lane is done. Before
// the o_proj units of an attention layer the whole warp stops: once every
// ring is drained it streams that layer's KV pages through the same shared
// memory (attn_stream), then resumes the weights.
__device__ __noinline__ void producer_warp(const ModelDesc& md, const StepDesc& sd, const Smem& sm, const CUtensorMap* tmk,
                              const CUtensorMap* tmv) {
  const int lane = threadIdx.x & 31;
  const int w = lane < kWarps ? lane : 0;
  const uint64_t pol = evict_first_policy();
  int gp = -1;
  uint32_t left = 0, tile = 0, sbl = 0, p = 0, kv_issued = 0;
  int nsb_s = 1, sb0 = 0, nsb = 1;
  const uint8_t* wsrc = nullptr;
  bool done = lane >= kWarps;
  int hold = -1;            // attention layer this lane stopped at
  int attn_done_upto = -1;  // last attention layer whose pages were streamed
  bool failed = false;
  volatile int32_t* err = md.err;
  uint64_t t_idle = 0;
  const int last_gp = md.has_mtp ? mtp_gp0(md) + 6 * md.n_draft - 1 : 4 * md.n_layers;
  for (uint32_t sweep = 0;; ++sweep) {
    // advance to the next phase with units for this lane's warp
    while (!done && left == 0 && hold < 0) {
      const int ngp = gp + 1;
      if (ngp > last_gp) { done = true; break; }
      const int ak = attn_key_before(md, ngp);
      if (ak >= 0 && ak > attn_done_upto) {
        hold = ak;
        break;
      }
      gp = ngp;
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
    if (__all_sync(0xffffffffu, done || hold >= 0)) {
      const int hl = __shfl_sync(0xffffffffu, hold, 0);
      if (hl < 0) break;  // every lane is done
      // every weight unit issued so far must be consumed before pages land in the ring
      bool ok = true;
      if (lane < kWarps && p > 0)
        ok = mbar_wait_bounded(sm.empty(w, (p - 1) % kRing), ((p - 1) / kRing) & 1u, md, sd.barrier_timeout_ns,
                               DEV_COPY_TIMEOUT);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) ok = attn_stream(md, sd, sm, hl < md.n_layers ? hl : md.n_layers, tmk, tmv, kv_issued, pol);
      if (!ok) { failed = true; break; }
      attn_done_upto = hl;
      if (lane < kWarps) hold = -1;
      continue;
    }
    bool issued = false;
    if (!done && left > 0) {
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
      continue;
    }
    // nothing could be issued: the math warps are behind; nap so that the
    // polling does not take issue slots from the math warps on this SMSP
    if (kProducerNapNs > 0) __nanosleep(kProducerNapNs);
    if ((sweep & 63u) == 63u) {
      // give up only on
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
  if (failed && lane < sd.attn_ng && sd.attn_spg > 0) {
    const AttnBuf ab = attn_buf(sm);
    const uint32_t spg = static_cast<uint32_t>(sd.attn_spg);
    for (uint32_t q = kv_issued > spg ? kv_issued - spg : 0; q < kv_issued; ++q)
      mbar_wait_bounded(ab.full + lane * spg + q % spg, (q / spg) & 1u, md, 50000000ull, DEV_COPY_TIMEOUT);
  }
}

// ------------------------------------------------------------- the kernel
// 9 warps: at most 168 registers each (three warps share a sub-partition).
__global__ void __launch_bounds__(kLaunchThreads, 1)
    mk_persistent(const ModelDesc* __restrict__ mdp, const StepDesc* __restrict__ sdp,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  __shared__ int sflag;
  const Smem sm{};
  const ModelDesc& md = *mdp;
  const StepDesc& sd = *sdp;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x < kWarps * kRing) {
    mbar_init(sm.bar(threadIdx.x / kRing, threadIdx.x % kRing), 1);
    mbar_init(sm.empty(threadIdx.x / kRing, threadIdx.x % kRing), 1);
  }
  if (threadIdx.x < kAttnMaxSlots) {
    const AttnBuf ab = attn_buf(sm);
    mbar_init(ab.full + threadIdx.x, 1);
    mbar_init(ab.empty + threadIdx.x, sd.attn_wpg > 0 ? sd.attn_wpg : 1);
  }
  mbar_fence_init();
  __syncthreads();
  if (warp == kWarps) {  // the producer warp
    producer_warp(md, sd, sm, &tm_k, &tm_v);
    return;
  }
  WarpCtx wc;
  wc.warp = warp;
  wc.lane = threadIdx.x & 31;
  wc.gid = blockIdx.x * kWarps + wc.warp;
  wc.c_pos = 0;
  wc.kv_pos = 0;

  int nbar = 0;
  // Phases: 0 embed; then per layer l: 1+5l input GEMM, 2+5l mixer,
  // 3+5l o_proj, 4+5l gate/up, 5+5l down; then lm_head; then verify. With an
  // MTP head, nine more per draft pass p: input rows, W_fc, input
  // projections, attention, o_proj, gate/up, down, draft lm_head, draft.
  const int n_main = 1 + 5 * md.n_layers + 2;
  const int n_phases = n_main + (md.has_mtp ? 9 * md.n_draft : 0);
  auto attention = [&](int layer, int mp) {
    if (!md.kv_q8) return attn_dispatch<false, true>(sd.attn_nq, sd.attn_jw, md, sd, layer, sm, wc, mp);
    if (md.dh % 128 == 0)
      return attn_dispatch<true, true>(sd.attn_nq, sd.attn_jw, md, sd, layer, sm, wc, mp);
    return attn_dispatch<true, false>(sd.attn_nq, sd.attn_jw, md, sd, layer, sm, wc, mp);
  };
  if (md.dbg_time && blockIdx.x == 0 && threadIdx.x == 0) md.dbg_time[0] = globaltimer();
  for (int ph = 0; ph < n_phases; ++ph) {
    bool ok = true;
    int gp = -1;
    if (ph == 0) {
      embed_phase(md, sd, wc);
    } else if (ph == n_main - 1) {
      verify_phase(md, sd, sm);
      if (!md.has_mtp) break;
    } else if (ph == n_main - 2) {
      gp = 4 * md.n_layers;
    } else if (ph < n_main) {
      const int l = (ph - 1) / 5, part = (ph - 1) % 5;
      if (part == 1) {
        if (md.layer[l].kind == MK_LAYER_GDN) gdn_phase(md, sd, l, wc, sm);
        else ok = attention(l, 0);
      } else {
        gp = 4 * l + (part == 0 ? 0 : part - 1);
      }
    } else {
      const int q = ph - n_main, mp = q / 9, part = q % 9;
      const int g0 = mtp_gp0(md) + 6 * mp;
      if (part == 0) mtp_input_phase(md, sd, mp, sm);
      else if (part <= 2) gp = g0 + part - 1;
      else if (part == 3) ok = attention(md.n_layers, mp);
      else if (part <= 7) gp = g0 + part - 2;
      else {
        draft_phase(md, sd, mp);
        if (mp + 1 == md.n_draft) break;  // nothing in the launch reads the last drafts
      }
    }
    if (gp >= 0) ok = gemm_dispatch(md, sd, gp, sm, wc);
    // a failed wait inside a phase still meets the barrier, which reports it
    bool synced = grid_sync(md, sd, nbar, &sflag);
    if (md.dbg_time && ph < n_main && blockIdx.x == 0 && threadIdx.x == 0) md.dbg_time[ph + 1] = globaltimer();
    if (!synced || !ok) break;
    if (gp >= 0 && is_top_gp(md, gp)) {
      const GemmDesc& g = gemm_desc(md, gp);
      if (make_sched(g.nsb, sd.R).S > 1) {  // sliced lm_head: scan the summed logits
        lm_argmax(md, sd, g, wc);
        synced = grid_sync(md, sd, nbar, &sflag);
        if (!synced) break;
      }
    }
  }
}

cudaError_t launch_persistent(const ModelDesc* md, const StepDesc* sd, int grid,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, cudaStream_t stream) {
  void* args[] = {const_cast<ModelDesc**>(&md), const_cast<StepDesc**>(&sd),
                  const_cast<CUtensorMap*>(tm_k), const_cast<CUtensorMap*>(tm_v)};
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
