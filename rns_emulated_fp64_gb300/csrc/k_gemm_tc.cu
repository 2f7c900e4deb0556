// Step 3: N exact residue matrix products on the 5th-generation tensor cores.
//
// [Q] "誤差のないINT8行列積(手順3)": per modulus, one integer product of the
// residue matrices, exact in INT32 because |r_a r_b| <= 128*128 = 2^14 and the
// inner dimension stays below 2^17.  sm_103a has no integer tcgen05 MMA, so
// the residues are held as FP16 (exact for integers up to 2048) and multiplied
// with tcgen05.mma kind::f16 into FP32 accumulators in tensor memory.  An FP32
// accumulator is exact while every partial sum is an integer below 2^24 in
// magnitude, so the k loop is cut into chunks and the accumulator is reduced
// between chunks ("lazy" reduction: only when it could otherwise overflow):
//
//  KIND 0 (mod-p output): 128x256 tiles.  The k loop is cut into
//    ceil(k-blocks / 15) chunks of at most 15 k-blocks, with lengths that
//    differ by at most one.  After each chunk (at most 960 terms, |partial| <=
//    134 + 960 * 2^14 < 2^24) the epilogue warps read
//    the accumulator, subtract the nearest multiple of p_l and write the small
//    remainder back; the next chunk accumulates on top of it.  Two jobs (tile x
//    modulus) are interleaved chunk by chunk, one per TMEM buffer, so the MMA
//    of one job runs while the other job's accumulator is being reduced.  The
//    final reduction is the canonical symmetric residue c_l, stored as int8.
//
//  KIND 1 (exact int32): 128x128 tiles.  Each chunk starts a fresh FP32
//    accumulator (ping-pong between two TMEM buffers); the epilogue converts it
//    to int32 and adds it to a running sum held in registers.  Outputs: the raw
//    int32 product (parity checks) and/or its row and column maxima (the bound
//    product of the accurate mode, where the 2-SM kernel below cannot be used).
//
//  k_gemm_tc2 (further down): the same mod-p product on CTA pairs with 256x256
//    tiles (the default), and the accurate-mode bound product in 4096-term
//    segments.
//
// Warp roles (192 threads, one CTA per SM, persistent over jobs):
//   warp 0     TMA producer: 128-byte-swizzled k-blocks of A and B into a
//              multi-stage shared-memory ring (mbarrier full/empty pairs).
//   warp 1     TMEM allocation; one elected thread issues tcgen05.mma and
//              tcgen05.commit.
//   warps 2-5  epilogue: tcgen05.ld / st on their 32-lane TMEM quarter.
// Every wait is bounded; on expiry the CTA records OS2_ERR_TIMEOUT, lets its
// copies and MMAs drain (again bounded), frees its TMEM and returns.
#include <cudaTypedefs.h>
#include <mutex>

#include "os2_internal.cuh"
#include "ptx.cuh"

using namespace os2ptx;

namespace {

constexpr int BM = 128;
constexpr int BK = 64;               // FP16 elements per k-block (128 bytes)
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s)

template <int KIND>
struct Cfg;
template <>
struct Cfg<0> {
  static constexpr int BN = 256, STAGES = 4, TMEM_COLS = 512;
};
template <>
struct Cfg<1> {
  static constexpr int BN = 128, STAGES = 6, TMEM_COLS = 256;
};

struct Sched {
  int m, n, kb_total;
  int tiles_m, tiles_n, tiles;
  int njobs;
  int chunk, nchunks;
};

__device__ __forceinline__ void job_coords(int job, const Sched &sp, int &l, int &tm, int &tn) {
  l = job / sp.tiles;
  int t = job - l * sp.tiles;
  constexpr int GM = 8;  // tile rows per raster group (L2 reuse of B tiles)
  int group = t / (GM * sp.tiles_n);
  int first = group * GM;
  int rows_in = min(GM, sp.tiles_m - first);
  int w = t - group * GM * sp.tiles_n;
  tm = first + w % rows_in;
  tn = w / rows_in;
}

// First k-block of chunk c: the kb_total k-blocks split into nchunks chunks
// whose lengths differ by at most one (each <= sp.chunk, since nchunks =
// ceil(kb_total / chunk)), so no chunk is much shorter than the epilogue work
// that overlaps it.
__device__ __forceinline__ int chunk_begin(const Sched &sp, int c) {
  return (int)((long long)c * sp.kb_total / sp.nchunks);
}

// The unit sequence every role walks: (job, chunk, TMEM buffer).
template <int KIND, typename F>
__device__ __forceinline__ void for_each_unit_of(const Sched &sp, int b, int G, F &&f) {
  const int cj = b < sp.njobs ? (sp.njobs - 1 - b) / G + 1 : 0;
  if (KIND == 0) {
    for (int q = 0; q < cj; q += 2) {
      const int nj = min(2, cj - q);
      for (int c = 0; c < sp.nchunks; c++)
        for (int s = 0; s < nj; s++)
          if (!f(b + (q + s) * G, c, s)) return;
    }
  } else {
    int u = 0;
    for (int q = 0; q < cj; q++)
      for (int c = 0; c < sp.nchunks; c++, u++)
        if (!f(b + q * G, c, u & 1)) return;
  }
}
template <int KIND, typename F>
__device__ __forceinline__ void for_each_unit(const Sched &sp, F &&f) {
  for_each_unit_of<KIND>(sp, (int)blockIdx.x, (int)gridDim.x, f);
}

__device__ __forceinline__ void set_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
              const Sched sp, const GemmConsts gc, void *__restrict__ out, int ldo,
              int32_t *__restrict__ rowmax, int32_t *__restrict__ colmax, int *status) {
  using C = Cfg<KIND>;
  constexpr int BN = C::BN, STAGES = C::STAGES;
  constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2;
  constexpr uint32_t IDESC = idesc_f16_f32(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  uint64_t *full = bars, *empty = bars + STAGES;
  uint64_t *acc_full = bars + 2 * STAGES, *acc_empty = acc_full + 2, *mma_done = acc_empty + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(mma_done + 1);
  volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_par = 0;  // per stage: ever used / parity of its last load
      for_each_unit<KIND>(sp, [&](int job, int c, int) -> bool {
        int l, tm, tn;
        job_coords(job, sp, l, tm, tn);
        const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
        for (int kb = kb0; kb < kb1; kb++) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, s_abort, kWaitLimit)) {
            *s_abort = 1;
            set_status(status, OS2_ERR_TIMEOUT);
            return false;
          }
          mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
          tma_load_3d(sA + stage * A_BYTES, &mapA, &full[stage], kb * BK, tm * BM, l);
          tma_load_3d(sB + stage * B_BYTES, &mapB, &full[stage], kb * BK, tn * BN, l);
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        return true;
      });
      // let every issued copy land before the CTA can exit
      for (int s = 0; s < STAGES; s++)
        if (used >> s & 1) {
          volatile int no_abort = 0;
          mbar_wait_bounded(&full[s], (last_par >> s) & 1, &no_abort, kWaitLimit);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t aphase[2] = {0, 0};
      for_each_unit<KIND>(sp, [&](int, int c, int buf) -> bool {
        if (!mbar_wait_bounded(&acc_empty[buf], aphase[buf] ^ 1, s_abort, kWaitLimit)) {
          *s_abort = 1;
          set_status(status, OS2_ERR_TIMEOUT);
          return false;
        }
        aphase[buf] ^= 1;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);
        const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
        for (int kb = kb0; kb < kb1; kb++) {
          if (!mbar_wait_bounded(&full[stage], phase, s_abort, kWaitLimit)) {
            *s_abort = 1;
            set_status(status, OS2_ERR_TIMEOUT);
            return false;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k128(smem_u32(sA + stage * A_BYTES));
          const uint64_t bd = sdesc_k128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 16; kk++) {
            const uint32_t acc = (kb > kb0 || kk > 0 || (KIND == 0 && c > 0)) ? 1u : 0u;
            umma_f16(d, ad + 2 * kk, bd + 2 * kk, IDESC, acc);  // +32 bytes along k
          }
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        umma_commit(&acc_full[buf]);
        return true;
      });
      umma_commit(mma_done);
      volatile int no_abort = 0;
      mbar_wait_bounded(mma_done, 0, &no_abort, kWaitLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    uint32_t aphase[2] = {0, 0};
    if (KIND == 0) {
      int8_t *outp = reinterpret_cast<int8_t *>(out);
      for_each_unit<KIND>(sp, [&](int job, int c, int buf) -> bool {
        // every lane waits (acquire), then the warp reconverges on one verdict
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], aphase[buf],
                                                                   s_abort, kWaitLimit));
        if (!ok) {
          *s_abort = 1;
          set_status(status, OS2_ERR_TIMEOUT);
          return false;
        }
        aphase[buf] ^= 1;
        tc_fence_after();
        int l, tm, tn;
        job_coords(job, sp, l, tm, tn);
        const float p = gc.p[l], invp = gc.invp[l];
        const uint32_t taddr = lane_base + (uint32_t)(buf * BN);
        if (c != sp.nchunks - 1) {
          // intermediate: subtract the nearest multiple of p, keep |r| <= ~0.52 p
#pragma unroll 1
          for (int g = 0; g < BN / 32; g++) {
            uint32_t v[32];
            tmem_ld32(taddr + g * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; i++) {
              float x = __uint_as_float(v[i]);
              v[i] = __float_as_uint(fmaf(-p, rintf(x * invp), x));
            }
            tmem_st32(taddr + g * 32, v);
          }
          tmem_wait_st();
        } else {
          // final: canonical symmetric residue, int8 store
          const float hi = gc.hi[l], lo = gc.lo[l];
          const int grow = tm * BM + r_in_tile;
          const int col0 = tn * BN;
          int8_t *dst = outp + ((size_t)l * sp.m + grow) * (size_t)ldo + col0;
#pragma unroll 1
          for (int g = 0; g < BN / 32; g++) {
            uint32_t v[32];
            tmem_ld32(taddr + g * 32, v);
            tmem_wait_ld();
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; i++) packed[i] = 0;
#pragma unroll
            for (int i = 0; i < 32; i++) {
              float x = __uint_as_float(v[i]);
              float r = fmaf(-p, rintf(x * invp), x);
              r = r > hi ? r - p : r;
              r = r < lo ? r + p : r;
              packed[i >> 2] |= ((uint32_t)(int)r & 0xFFu) << (8 * (i & 3));
            }
            if (grow < sp.m && OS2_DBG_GUARD(l < gc.N && sp.n <= ldo, status)) {
              const int cb = col0 + g * 32;
              if (cb + 32 <= sp.n) {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + g * 32);
                d4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                d4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              } else {
                for (int i = 0; i < 32 && cb + i < sp.n; i++)
                  dst[g * 32 + i] = (int8_t)((packed[i >> 2] >> (8 * (i & 3))) & 0xFFu);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        return true;
      });
    } else {
      int32_t *outp = reinterpret_cast<int32_t *>(out);
      int acc[BN];
#pragma unroll
      for (int i = 0; i < BN; i++) acc[i] = 0;
      for_each_unit<KIND>(sp, [&](int job, int c, int buf) -> bool {
        // every lane waits (acquire), then the warp reconverges on one verdict
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], aphase[buf],
                                                                   s_abort, kWaitLimit));
        if (!ok) {
          *s_abort = 1;
          set_status(status, OS2_ERR_TIMEOUT);
          return false;
        }
        aphase[buf] ^= 1;
        tc_fence_after();
        const uint32_t taddr = lane_base + (uint32_t)(buf * BN);
#pragma unroll
        for (int g = 0; g < BN / 32; g++) {
          uint32_t v[32];
          tmem_ld32(taddr + g * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i++) {
            int x = __float2int_rn(__uint_as_float(v[i]));
            acc[g * 32 + i] = (c == 0) ? x : acc[g * 32 + i] + x;
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        if (c == sp.nchunks - 1) {
          int l, tm, tn;
          job_coords(job, sp, l, tm, tn);
          const int grow = tm * BM + r_in_tile;
          const int col0 = tn * BN;
          if (outp && grow < sp.m) {
            int32_t *dst = outp + ((size_t)l * sp.m + grow) * (size_t)ldo + col0;
            if (col0 + BN <= sp.n) {
#pragma unroll
              for (int i = 0; i < BN; i += 4)
                *reinterpret_cast<int4 *>(dst + i) = make_int4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < BN; i++)
                if (col0 + i < sp.n) dst[i] = acc[i];
            }
          }
          if (rowmax) {
            int mx = 0;
#pragma unroll
            for (int i = 0; i < BN; i++) mx = max(mx, acc[i]);
            if (grow < sp.m) atomicMax(&rowmax[grow], mx);
          }
          if (colmax) {
#pragma unroll
            for (int i = 0; i < BN; i++) {
              int v = __reduce_max_sync(0xffffffffu, acc[i]);
              if (lane == 0 && col0 + i < sp.n) atomicMax(&colmax[col0 + i], v);
            }
          }
        }
        return true;
      });
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}


// -------------------------------------------------------------------------
// 2-SM variant of KIND 0: a CTA pair (cluster of 2) computes a 256x256 tile
// with tcgen05.mma.cta_group::2 issued by the even CTA.  Each CTA loads 128
// rows of the A tile and 128 rows of the B tile (its half of N) into a ring
// of kStages2 stages of kKbStage2 k-blocks; both CTAs' copies complete on the
// even CTA's "full" barrier,
// the MMA commits are multicast to both CTAs' "empty" and "accumulator full"
// barriers, and both CTAs' epilogues release an accumulator on the even
// CTA's "accumulator empty" barrier.  Each CTA's TMEM holds its 128 rows x
// 256 columns of the two interleaved jobs, reduced mod p like the single-SM
// kernel's (with FMA-only rounding, see above).  Chunks are counted in stages:
// at most 7 stages of two k-blocks (896 terms) between reductions.  Per SM
// this halves the B-tile traffic of the single-SM kernel.
// A stage holds two k-blocks (128 terms): one operand wait, fence and commit
// per eight MMAs.  Measured at 8192^3 with 16 moduli, the same shared memory
// cut into 6 or 7 stages of one k-block ran 4.5 % slower.
constexpr int kKbStage2 = 2;  // k-blocks per stage
constexpr int kStages2 = 3;
constexpr int kHalf = 128;
constexpr int BK2 = 2 * BK;  // terms per stage of the int8-plane variant

// ---------------------------------------------- 2-SM epilogue arithmetic
// Accumulators hold exact integers |x| < 2^24.  Adding 1.5 * 2^23 rounds a
// value of magnitude < 2^22 to an integer (ties to even) in the FMA's single
// rounding, so x - p * round(x * fl(1/p)) takes three full-rate FP32 ops.
constexpr float kRound = 12582912.0f;  // 1.5 * 2^23

// An exact integer congruent to x mod p, of magnitude <= p/2 + 1:
// |x * fl(1/p) - x / p| <= |x| * 2^-32 < 2^-8 for 128 < p <= 256.
__device__ __forceinline__ float reduce_near(float x, float p, float invp) {
  const float q = fmaf(x, invp, kRound) - kRound;
  return fmaf(-p, q, x);
}

// The low byte of the symmetric residue of x.  After one step |r| <= p/2 + 1;
// a second step moves the extremes +-(p+1)/2 of an odd p into range and leaves
// the rest; for p = 256 the values +-128 share the byte 0x80.  r + 1.5 * 2^23
// is exact and carries r mod 256 in its low byte.
__device__ __forceinline__ uint32_t residue_byte(float x, float p, float invp) {
  const float r = reduce_near(reduce_near(x, p, invp), p, invp);
  return __float_as_uint(r + kRound);
}

// Low bytes of a, b, c, d packed into one word (a in the lowest byte).
__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Accurate-mode bound product on the 2-SM kernel (BOUND = 1): one launch per
// segment of at most 4096 terms, whose FP32 sums (Abar, Bbar <= 64, so each
// product <= 2^12 and a segment's sum <= 2^24) are exact.  Segments after the
// first add the int32 partial sums of the earlier ones; the last takes the
// row and column maxima.
struct BoundSeg {
  int kb_begin;          // first stage of the segment
  int first, last;       // segment flags
  int32_t *partial;      // int32 [m][ldp] partial sums between segments
  int ldp;
  int32_t *rowmax, *colmax;
};

// Bound-segment epilogue: this thread's row `grow` of the tile, 256 columns
// from col0, read from TMEM as exact FP32 integers.  Rows and columns past the
// matrix hold 0 (zero-filled operand tiles), which never changes a maximum.
// The partial sums move as 16-byte vectors (ldp is a multiple of 4), and a
// group's partial loads are issued before its TMEM load is waited on.
__device__ __forceinline__ void bound_epilogue(uint32_t taddr, int grow, int col0, int lane,
                                               const Sched &sp, const BoundSeg &bs, int *status) {
  const bool row_ok =
      grow < sp.m && OS2_DBG_GUARD((bs.first && bs.last) || sp.n <= bs.ldp, status);
  int rmax = 0;
#pragma unroll 1
  for (int g = 0; g < 256 / 32; g++) {
    const int cb = col0 + g * 32;
    const bool full = cb + 32 <= sp.n;
    int4 *prow = reinterpret_cast<int4 *>(bs.partial + (size_t)(row_ok ? grow : 0) * bs.ldp + cb);
    int4 pv[8];
    if (!bs.first && row_ok && full) {
#pragma unroll
      for (int q = 0; q < 8; q++) pv[q] = prow[q];
    }
    uint32_t v[32];
    tmem_ld32(taddr + g * 32, v);
    tmem_wait_ld();
    int x[32];
#pragma unroll
    for (int i = 0; i < 32; i++) x[i] = __float2int_rn(__uint_as_float(v[i]));
    int *ps = reinterpret_cast<int *>(prow);
    if (!bs.first && row_ok) {
      if (full) {
#pragma unroll
        for (int q = 0; q < 8; q++) {
          x[4 * q] += pv[q].x;
          x[4 * q + 1] += pv[q].y;
          x[4 * q + 2] += pv[q].z;
          x[4 * q + 3] += pv[q].w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; i++)
          if (cb + i < sp.n) x[i] += ps[i];
      }
    }
    if (!bs.last) {
      if (row_ok) {
        if (full) {
#pragma unroll
          for (int q = 0; q < 8; q++)
            prow[q] = make_int4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; i++)
            if (cb + i < sp.n) ps[i] = x[i];
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) {
        rmax = max(rmax, x[i]);
        const int cm = __reduce_max_sync(0xffffffffu, x[i]);  // over the warp's 32 rows
        if (lane == i && cb + i < sp.n) atomicMax(&bs.colmax[cb + i], cm);
      }
    }
  }
  if (bs.last && row_ok) atomicMax(&bs.rowmax[grow], rmax);
}

// int8-plane variant (I8 = 1): the residue planes come from HBM as int8 (half
// the bytes of FP16); TMA copies each CTA's 128 rows x 128 k of A and of B into
// a ring of int8 stages (unswizzled 128-byte rows, completion on the CTA's own
// barrier), and four more warps widen a stage into the FP16 operand ring the
// MMAs read (same 128-byte-swizzled layout as the TMA writes in the FP16
// kernel): 1024 + (r + 128) is the FP16 with bit pattern 0x64 followed by the
// byte r ^ 0x80, and one packed FP16 add of -1152 leaves r exactly.  Both CTAs'
// converters (eight warps each) arrive on the even CTA's "operand full"
// barrier; the MMA's commit is multicast to both CTAs' "operand empty"
// barriers as before.
constexpr int kStages2I8 = 2;      // FP16 operand stages of the int8 variant
constexpr int kRawStages2 = 3;     // int8 stages
constexpr int kConvThreads = 256;  // converter warps 6-13

// k-blocks per FP16 operand stage: the int8-plane variant converts two at a time
template <int I8>
constexpr int kb_per_stage2() {
  return I8 ? 2 : kKbStage2;
}

template <int I8>
constexpr size_t smem2_bytes() {
  return 1024 + (size_t)(I8 ? kStages2I8 : kStages2) * kb_per_stage2<I8>() * 2 * kHalf * BK * 2 +
         (I8 ? (size_t)kRawStages2 * 2 * kHalf * BK2 : 0) + 256;
}

__device__ __forceinline__ uint32_t hadd2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Exact FP16 of the four int8 residues of a word: [r0 r1] and [r2 r3].
__device__ __forceinline__ void widen_exact(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t x = w ^ 0x80808080u;
  lo = hadd2_bits(__byte_perm(x, 0x64646464u, 0x4140), 0xE480E480u);  // - 1152
  hi = hadd2_bits(__byte_perm(x, 0x64646464u, 0x4342), 0xE480E480u);
}

template <int BOUND, int I8 = 0>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(I8 ? kThreads + kConvThreads : kThreads, 1)
    k_gemm_tc2(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const Sched sp, const GemmConsts gc, int8_t *__restrict__ out, int ldo,
               const BoundSeg bs, int *status) {
  constexpr int BN = 256, STAGES = I8 ? kStages2I8 : kStages2;
  constexpr int KPS = kb_per_stage2<I8>();  // k-blocks per FP16 stage
  constexpr int RSTAGES = I8 ? kRawStages2 : 0;
  constexpr uint32_t HALF = kHalf * BK * 2;  // one k-block of 128 rows
  constexpr uint32_t A_BYTES = KPS * HALF, B_BYTES = KPS * HALF;
  constexpr uint32_t RAW_HALF = kHalf * BK2;  // int8 stage: 128 rows x 128 bytes of A (or B)
  constexpr uint32_t RAW_BYTES = 2 * RAW_HALF;
  constexpr uint32_t IDESC = idesc_f16_f32(2 * kHalf, BN);
  constexpr uint32_t TMEM_COLS = 512;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * A_BYTES;
  uint8_t *sRaw = sB + STAGES * B_BYTES;  // int8 stages (I8)
  uint64_t *bars = reinterpret_cast<uint64_t *>(sRaw + RSTAGES * RAW_BYTES);
  uint64_t *full = bars, *empty = bars + STAGES;
  uint64_t *acc_full = bars + 2 * STAGES, *acc_empty = acc_full + 2, *mma_done = acc_empty + 2;
  uint64_t *rfull = mma_done + 1, *rempty = rfull + RSTAGES;  // int8 ring (I8)
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(rempty + RSTAGES);
  volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(&full[s], I8 ? 2 * kConvThreads : 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < RSTAGES; s++) {
      mbar_init(&rfull[s], 1);
      mbar_init(&rempty[s], kConvThreads);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kEpiThreads);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) {
    tmem_alloc2(s_tmem, TMEM_COLS);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive / copy
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  if (I8 && warp == 0) {
    // ------------------------------------------------------------ int8 copies
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0, used = 0, last_par = 0;
      for_each_unit_of<0>(sp, pair, npairs, [&](int job, int c, int) -> bool {
        int l, tm, tn;
        job_coords(job, sp, l, tm, tn);
        const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
        for (int kb = kb0; kb < kb1; kb++) {
          if (!mbar_wait_bounded(&rempty[rs], rph ^ 1, s_abort, kWaitLimit)) {
            *s_abort = 1;
            set_status(status, OS2_ERR_TIMEOUT);
            return false;
          }
          mbar_arrive_expect_tx(&rfull[rs], RAW_BYTES);
          // a stage past the last k-block reads zeros (out-of-range box)
          tma_load_3d(sRaw + rs * RAW_BYTES, &mapA, &rfull[rs], kb * BK2,
                      tm * 2 * kHalf + (int)rank * kHalf, l);
          tma_load_3d(sRaw + rs * RAW_BYTES + RAW_HALF, &mapB, &rfull[rs], kb * BK2,
                      tn * BN + (int)rank * kHalf, l);
          used |= 1u << rs;
          last_par = (last_par & ~(1u << rs)) | (rph << rs);
          if (++rs == RSTAGES) {
            rs = 0;
            rph ^= 1;
          }
        }
        return true;
      });
      for (int s = 0; s < RSTAGES; s++)
        if (used >> s & 1) {
          volatile int no_abort = 0;
          mbar_wait_bounded(&rfull[s], (last_par >> s) & 1, &no_abort, kWaitLimit);
        }
    }
  } else if (I8 && warp >= 2 + kEpiThreads / 32) {
    // ------------------------------------------------------------ int8 -> FP16
    // thread ct widens 16-byte chunks q = ct + 256 i of the stage (A's 1024
    // chunks, then B's): the 8 lanes of a quarter-warp take the 8 chunks of one
    // 128-byte row, and each chunk becomes two 16-byte FP16 chunks of k-block
    // (chunk / 4) of the swizzled operand tile
    const int ct = threadIdx.x - kThreads;
    uint32_t full_leader[STAGES];
#pragma unroll
    for (int s2 = 0; s2 < STAGES; s2++) full_leader[s2] = mapa_shared(smem_u32(&full[s2]), 0);
    int rs = 0, fs = 0;
    uint32_t rph = 0, fph = 0;
    for_each_unit_of<0>(sp, pair, npairs, [&](int, int c, int) -> bool {
      const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
      for (int kb = kb0; kb < kb1; kb++) {
        const bool ok =
            mbar_wait_bounded(&rfull[rs], rph, s_abort, kWaitLimit) &&
            mbar_wait_cluster_bounded(&empty[fs], fph ^ 1, s_abort, kWaitLimit);
        if (!ok) {
          *s_abort = 1;
          set_status(status, OS2_ERR_TIMEOUT);
          return false;
        }
        const uint32_t rbase = smem_u32(sRaw + rs * RAW_BYTES);
        const uint32_t abase = smem_u32(sA + fs * A_BYTES), bbase = smem_u32(sB + fs * B_BYTES);
#pragma unroll
        for (int i = 0; i < (int)(RAW_BYTES / 16) / kConvThreads; i++) {
          const int q = i * kConvThreads + ct;
          const int op = q >> 10, row = (q >> 3) & 127, cc = q & 7;
          uint4 w;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(rbase + op * RAW_HALF + row * 128 + cc * 16));
          uint32_t h[8];
          widen_exact(w.x, h[0], h[1]);
          widen_exact(w.y, h[2], h[3]);
          widen_exact(w.z, h[4], h[5]);
          widen_exact(w.w, h[6], h[7]);
          const uint32_t rowa = (op ? bbase : abase) + (cc >> 2) * HALF + (row >> 3) * 1024 +
                                (row & 7) * 128;
          const int j0 = 2 * (cc & 3);
          const uint32_t d0 = rowa + ((j0 ^ (row & 7)) << 4);
          const uint32_t d1 = rowa + (((j0 + 1) ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d0), "r"(h[0]), "r"(h[1]),
                       "r"(h[2]), "r"(h[3])
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d1), "r"(h[4]), "r"(h[5]),
                       "r"(h[6]), "r"(h[7])
                       : "memory");
        }
        // the FP16 stage, written through the generic proxy, is read by the
        // tensor cores of the pair
        asm volatile("fence.proxy.async;" ::: "memory");
        mbar_arrive_cluster(full_leader[fs]);
        mbar_arrive(&rempty[rs]);
        if (++rs == RSTAGES) {
          rs = 0;
          rph ^= 1;
        }
        if (++fs == STAGES) {
          fs = 0;
          fph ^= 1;
        }
      }
      return true;
    });
  } else if (warp == 0) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_par = 0;
      for_each_unit_of<0>(sp, pair, npairs, [&](int job, int c, int) -> bool {
        int l, tm, tn;
        job_coords(job, sp, l, tm, tn);
        const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
        for (int kb = kb0; kb < kb1; kb++) {
          if (!mbar_wait_cluster_bounded(&empty[stage], phase ^ 1, s_abort, kWaitLimit)) {
            *s_abort = 1;
            set_status(status, OS2_ERR_TIMEOUT);
            return false;
          }
          const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (A_BYTES + B_BYTES));
          // a stage past the last k-block reads zeros (out-of-range box)
          const int kx = (BOUND ? bs.kb_begin + kb : kb) * (KPS * BK);
#pragma unroll
          for (int h = 0; h < KPS; h++) {
            tma_load_3d_pair(sA + stage * A_BYTES + h * HALF, &mapA, fbar, kx + h * BK,
                             tm * 2 * kHalf + (int)rank * kHalf, l);
            tma_load_3d_pair(sB + stage * B_BYTES + h * HALF, &mapB, fbar, kx + h * BK,
                             tn * BN + (int)rank * kHalf, l);
          }
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        return true;
      });
      if (leader)
        for (int s = 0; s < STAGES; s++)
          if (used >> s & 1) {
            volatile int no_abort = 0;
            mbar_wait_cluster_bounded(&full[s], (last_par >> s) & 1, &no_abort, kWaitLimit);
          }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t aphase[2] = {0, 0};
      for_each_unit_of<0>(sp, pair, npairs, [&](int, int c, int buf) -> bool {
        if (!mbar_wait_cluster_bounded(&acc_empty[buf], aphase[buf] ^ 1, s_abort, kWaitLimit)) {
          *s_abort = 1;
          set_status(status, OS2_ERR_TIMEOUT);
          return false;
        }
        aphase[buf] ^= 1;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * BN);
        const int kb0 = chunk_begin(sp, c), kb1 = chunk_begin(sp, c + 1);
        for (int kb = kb0; kb < kb1; kb++) {
          if (!mbar_wait_cluster_bounded(&full[stage], phase, s_abort, kWaitLimit)) {
            *s_abort = 1;
            set_status(status, OS2_ERR_TIMEOUT);
            return false;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < KPS; h++) {
            const uint64_t ad = sdesc_k128(smem_u32(sA + stage * A_BYTES + h * HALF));
            const uint64_t bd = sdesc_k128(smem_u32(sB + stage * B_BYTES + h * HALF));
#pragma unroll
            for (int kk = 0; kk < BK / 16; kk++) {
              const uint32_t acc = (kb > kb0 || h > 0 || kk > 0 || c > 0) ? 1u : 0u;
              umma2_f16(d, ad + 2 * kk, bd + 2 * kk, IDESC, acc);
            }
          }
          umma2_commit_mc(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        umma2_commit_mc(&acc_full[buf], 0x3);
        return true;
      });
      umma2_commit_mc(mma_done, 0x1);
      volatile int no_abort = 0;
      mbar_wait_bounded(mma_done, 0, &no_abort, kWaitLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t empty_leader[2] = {mapa_shared(smem_u32(&acc_empty[0]), 0),
                                      mapa_shared(smem_u32(&acc_empty[1]), 0)};
    uint32_t aphase[2] = {0, 0};
    for_each_unit_of<0>(sp, pair, npairs, [&](int job, int c, int buf) -> bool {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster_bounded(&acc_full[buf], aphase[buf],
                                                                         s_abort, kWaitLimit));
      if (!ok) {
        *s_abort = 1;
        set_status(status, OS2_ERR_TIMEOUT);
        return false;
      }
      aphase[buf] ^= 1;
      tc_fence_after();
      int l, tm, tn;
      job_coords(job, sp, l, tm, tn);
      const float p = gc.p[l], invp = gc.invp[l];
      const uint32_t taddr = lane_base + (uint32_t)(buf * BN);
      if (BOUND) {
        bound_epilogue(taddr, tm * 2 * kHalf + (int)rank * kHalf + r_in_tile, tn * BN, lane, sp,
                       bs, status);
      } else if (c != sp.nchunks - 1) {
        // intermediate chunk: reduce in place (|r| <= p/2 + 1 carries into the next chunk)
#pragma unroll 1
        for (int g = 0; g < BN / 32; g++) {
          uint32_t v[32];
          tmem_ld32(taddr + g * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i++)
            v[i] = __float_as_uint(reduce_near(__uint_as_float(v[i]), p, invp));
          tmem_st32(taddr + g * 32, v);
        }
        tmem_wait_st();
      } else {
        // final chunk: canonical symmetric residues as int8
        const int grow = tm * 2 * kHalf + (int)rank * kHalf + r_in_tile;
        const int col0 = tn * BN;
        int8_t *dst = out + ((size_t)l * sp.m + grow) * (size_t)ldo + col0;
#pragma unroll 1
        for (int g = 0; g < BN / 32; g++) {
          uint32_t v[32];
          tmem_ld32(taddr + g * 32, v);
          tmem_wait_ld();
          uint32_t packed[8];
#pragma unroll
          for (int i = 0; i < 8; i++)
            packed[i] = pack4(residue_byte(__uint_as_float(v[4 * i]), p, invp),
                              residue_byte(__uint_as_float(v[4 * i + 1]), p, invp),
                              residue_byte(__uint_as_float(v[4 * i + 2]), p, invp),
                              residue_byte(__uint_as_float(v[4 * i + 3]), p, invp));
          if (grow < sp.m && OS2_DBG_GUARD(l < gc.N && sp.n <= ldo, status)) {
            const int cb = col0 + g * 32;
            if (cb + 32 <= sp.n) {
              uint4 *d4 = reinterpret_cast<uint4 *>(dst + g * 32);
              d4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              d4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; i++)  // static indices keep `packed` in registers
                if (cb + i < sp.n) dst[g * 32 + i] = (int8_t)((packed[i >> 2] >> (8 * (i & 3))) & 0xFFu);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(empty_leader[buf]);
      return true;
    });
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory or TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc2(tmem_base, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// FP16 planes [nplanes][plane_rows][kp], of which the first `rows` rows are
// mapped; box = 64 (k) x box_rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int kp, int rows, int nplanes, int box_rows,
              int plane_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kp, (cuuint64_t)rows, (cuuint64_t)nplanes};
  cuuint64_t strides[2] = {(cuuint64_t)kp * 2, (cuuint64_t)kp * 2 * (cuuint64_t)plane_rows};
  cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int KIND>
cudaError_t launch(int m, int n, int kp, const void *RA, const void *RB, int nplanes, void *out,
                   int ldo, int32_t *rowmax, int32_t *colmax, int prod_bound_log2,
                   const Os2Tables *t, int *status, cudaStream_t s, int b_plane_rows) {
  using C = Cfg<KIND>;
  constexpr size_t smem = 1024 + (size_t)C::STAGES * (BM + C::BN) * BK * 2 + 256;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_gemm_tc<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb;
  if (!make_map(&ma, RA, kp, m, nplanes, BM, m) ||
      !make_map(&mb, RB, kp, n, nplanes, C::BN, b_plane_rows))
    return cudaErrorInvalidValue;
  Sched sp;
  sp.m = m;
  sp.n = n;
  sp.kb_total = kp / BK;
  sp.tiles_m = (m + BM - 1) / BM;
  sp.tiles_n = (n + C::BN - 1) / C::BN;
  sp.tiles = sp.tiles_m * sp.tiles_n;
  sp.njobs = sp.tiles * nplanes;
  // k-blocks per chunk keep every FP32 partial sum an exact integer below 2^24
  // (KIND 0 also carries a reduced remainder of magnitude <= 0.52 p + 1 <= 135).
  const long long cap = (1LL << 24) - (KIND == 0 ? 135 : 0);
  const long long per_block = (long long)BK << prod_bound_log2;
  sp.chunk = (int)(cap / per_block);
  if (sp.chunk < 1) return cudaErrorInvalidValue;
  sp.nchunks = (sp.kb_total + sp.chunk - 1) / sp.chunk;
  if (sp.njobs == 0 || sp.nchunks == 0) return cudaSuccess;
  const int grid = std::min(os2_sm_count(), sp.njobs);
  GemmConsts gc = t ? t->gemm : GemmConsts{};
  k_gemm_tc<KIND><<<grid, kThreads, smem, s>>>(ma, mb, sp, gc, out, ldo, rowmax, colmax, status);
  return cudaGetLastError();
}

template <int BOUND, int I8 = 0>
cudaError_t set_smem2() {
  constexpr size_t smem = smem2_bytes<I8>();
  static_assert(smem <= 227 * 1024, "shared memory of the 2-SM kernel");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_gemm_tc2<BOUND, I8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  return attr_err;
}

// int8 planes [nplanes][plane_rows][kp] bytes, of which the first `rows` rows
// are mapped; box = 128 (k) x 128 rows x 1, no swizzle.
bool make_map_i8(CUtensorMap *map, const void *base, int kp, int rows, int nplanes,
                 int plane_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kp, (cuuint64_t)rows, (cuuint64_t)nplanes};
  cuuint64_t strides[2] = {(cuuint64_t)kp, (cuuint64_t)kp * (cuuint64_t)plane_rows};
  cuuint32_t box[3] = {(cuuint32_t)BK2, (cuuint32_t)kHalf, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

Sched sched2(int m, int n, int kb_total, int nplanes) {
  Sched sp;
  sp.m = m;
  sp.n = n;
  sp.kb_total = kb_total;
  sp.tiles_m = (m + 2 * kHalf - 1) / (2 * kHalf);
  sp.tiles_n = (n + 255) / 256;
  sp.tiles = sp.tiles_m * sp.tiles_n;
  sp.njobs = sp.tiles * nplanes;
  return sp;
}

// i8: RA, RB are int8 planes (the int8-plane variant), else FP16 planes.
cudaError_t launch2(int m, int n, int kp, const void *RA, const void *RB, int nplanes, void *out,
                    int ldo, const Os2Tables *t, int *status, cudaStream_t s, int b_plane_rows,
                    bool i8 = false) {
  const size_t smem = i8 ? smem2_bytes<1>() : smem2_bytes<0>();
  cudaError_t attr_err = i8 ? set_smem2<0, 1>() : set_smem2<0>();
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb;
  const bool maps = i8 ? make_map_i8(&ma, RA, kp, m, nplanes, m) &&
                             make_map_i8(&mb, RB, kp, n, nplanes, b_plane_rows)
                       : make_map(&ma, RA, kp, m, nplanes, kHalf, m) &&
                             make_map(&mb, RB, kp, n, nplanes, kHalf, b_plane_rows);
  if (!maps) return cudaErrorInvalidValue;
  // the 2-SM kernel counts k in stages of kps k-blocks
  const int kps = i8 ? kb_per_stage2<1>() : kb_per_stage2<0>();
  Sched sp = sched2(m, n, (kp / BK + kps - 1) / kps, nplanes);
  sp.chunk = (int)(((1LL << 24) - 135) / ((long long)(kps * BK) << 14));
  sp.nchunks = (sp.kb_total + sp.chunk - 1) / sp.chunk;
  if (sp.njobs == 0 || sp.nchunks == 0) return cudaSuccess;
  const int pairs = std::min(std::max(os2_sm_count() / 2, 1), sp.njobs);
  GemmConsts gc = t ? t->gemm : GemmConsts{};
  if (i8)
    k_gemm_tc2<0, 1><<<2 * pairs, kThreads + kConvThreads, smem, s>>>(
        ma, mb, sp, gc, reinterpret_cast<int8_t *>(out), ldo, BoundSeg{}, status);
  else
    k_gemm_tc2<0><<<2 * pairs, kThreads, smem, s>>>(ma, mb, sp, gc,
                                                    reinterpret_cast<int8_t *>(out), ldo,
                                                    BoundSeg{}, status);
  return cudaGetLastError();
}

// Accurate-mode bound product (magnitude planes <= 64) with fused row and
// column maxima on the 2-SM kernel, in segments of at most 64 k-blocks.
cudaError_t launch2_bound(int m, int n, int kp, const void *RA, const void *RB, int32_t *partial,
                          int ldp, int32_t *rowmax, int32_t *colmax, int *status,
                          cudaStream_t s) {
  constexpr size_t smem = smem2_bytes<0>();
  constexpr int kps = kb_per_stage2<0>();
  constexpr int kSegMax = (int)((1LL << 24) / ((long long)(kps * BK) << 12));  // 4096 terms
  cudaError_t attr_err = set_smem2<1>();
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap ma, mb;
  if (!make_map(&ma, RA, kp, m, 1, kHalf, m) || !make_map(&mb, RB, kp, n, 1, kHalf, n))
    return cudaErrorInvalidValue;
  const int kb_all = (kp / BK + kps - 1) / kps;
  const int segs = (kb_all + kSegMax - 1) / kSegMax;
  if (segs > 1 && (!partial || ldp < n || ldp % 4 != 0 ||
                   (reinterpret_cast<uintptr_t>(partial) & 15)))
    return cudaErrorInvalidValue;
  for (int g = 0; g < segs; g++) {
    const int kb0 = (int)((long long)g * kb_all / segs), kb1 = (int)((long long)(g + 1) * kb_all / segs);
    Sched sp = sched2(m, n, kb1 - kb0, 1);
    sp.chunk = sp.kb_total;
    sp.nchunks = 1;
    if (sp.njobs == 0 || sp.kb_total == 0) return cudaSuccess;
    const int pairs = std::min(std::max(os2_sm_count() / 2, 1), sp.njobs);
    const BoundSeg bs{kb0, g == 0, g == segs - 1, partial, ldp, rowmax, colmax};
    k_gemm_tc2<1><<<2 * pairs, kThreads, smem, s>>>(ma, mb, sp, GemmConsts{}, nullptr, 0, bs,
                                                    status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_tc(int kind, int m, int n, int kp, const void *RA, const void *RB,
                           int nplanes, void *out, int ldo, int32_t *rowmax, int32_t *colmax,
                           int prod_bound_log2, const Os2Tables *t, int *status, cudaStream_t s,
                           int b_plane_rows) {
  if (m <= 0 || n <= 0 || kp <= 0) return cudaSuccess;
  if (b_plane_rows <= 0) b_plane_rows = n;
  if (b_plane_rows < n) return cudaErrorInvalidValue;
  if (kind == 2) return launch2(m, n, kp, RA, RB, nplanes, out, ldo, t, status, s, b_plane_rows);
  if (kind == 3)
    return launch2(m, n, kp, RA, RB, nplanes, out, ldo, t, status, s, b_plane_rows, true);
  if (kind == 0)
    return launch<0>(m, n, kp, RA, RB, nplanes, out, ldo, rowmax, colmax, prod_bound_log2, t,
                     status, s, b_plane_rows);
  return launch<1>(m, n, kp, RA, RB, nplanes, out, ldo, rowmax, colmax, prod_bound_log2, t,
                   status, s, b_plane_rows);
}

cudaError_t launch_gemm_bound2(int m, int n, int kp, const void *RA, const void *RB,
                               int32_t *partial, int ldp, int32_t *rowmax, int32_t *colmax,
                               int *status, cudaStream_t s) {
  if (m <= 0 || n <= 0 || kp <= 0) return cudaSuccess;
  return launch2_bound(m, n, kp, RA, RB, partial, ldp, rowmax, colmax, status, s);
}
