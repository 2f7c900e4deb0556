// Device helpers shared by the step 1 and step 2 kernels: decoding of
// binary64 / binary32 entries, paired loads, the status word and the row sets
// the kernels walk (A's rows, then B's columns as rows of B^T).
#pragma once
#include <cuda_fp16.h>
#include <limits.h>

#include "os2_internal.cuh"

namespace os2dev {

struct Dec {
  uint64_t mant;  // |x| = mant * 2^ex2
  int ex2;
  uint32_t neg;
  bool nonfinite;
};

__device__ __forceinline__ Dec decode(double x) {
  uint64_t b = (uint64_t)__double_as_longlong(x);
  int bexp = (int)((b >> 52) & 0x7FF);
  Dec d;
  d.neg = (uint32_t)(b >> 63);
  d.nonfinite = bexp == 0x7FF;
  d.mant = b & 0xFFFFFFFFFFFFFull;
  if (bexp) d.mant |= 1ull << 52;
  else bexp = 1;
  d.ex2 = bexp - 1075;
  if (d.nonfinite) d.mant = 0;
  return d;
}

__device__ __forceinline__ Dec decode(float x) {
  const uint32_t b = __float_as_uint(x);
  int bexp = (int)((b >> 23) & 0xFF);
  Dec d;
  d.neg = b >> 31;
  d.nonfinite = bexp == 0xFF;
  d.mant = b & 0x7FFFFFu;
  if (bexp) d.mant |= 1ull << 23;
  else bexp = 1;
  d.ex2 = bexp - 150;
  if (d.nonfinite) d.mant = 0;
  return d;
}

// Two consecutive entries through one vector load (aligned to 2 * sizeof(T)).
__device__ __forceinline__ void load2(const double *p, double &a, double &b) {
  const double2 v = __ldg(reinterpret_cast<const double2 *>(p));
  a = v.x;
  b = v.y;
}
__device__ __forceinline__ void load2(const float *p, float &a, float &b) {
  const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
  a = v.x;
  b = v.y;
}

__device__ __forceinline__ void set_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

struct RowSet {
  const void *X;    // double or float entries, row-major
  long ldx;
  int rows;
  int32_t *e;       // exponents (out for scale, in for residues)
  int32_t *E;       // accurate mode: exponent bounds (out)
  __half *planes;   // residue planes [N][prow][kp] (first `rows` rows written) or the
                    // magnitude plane [rows][kp]
  long prow;        // rows from one residue plane to the next (>= rows)
};

}  // namespace os2dev
