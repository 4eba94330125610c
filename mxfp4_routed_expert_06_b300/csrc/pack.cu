// pack.cu -- canonical MXFP4 -> packed tile layout (lossless byte permutation).
//
// The pages' engine multiplies directly on the nibbles ("kimi-k3-in-c deep dive", "four
// reductions", reduction 1) and calls the nibble order a convention that is silently wrong if
// flipped.  The canonical order (element 2i in the low nibble) already pairs the two columns
// that one tensor-core fragment register holds, so packing only moves whole bytes: each
// 16-byte lane chunk of a tile gathers the bytes one lane's mma.m16n8k16 A fragments need,
// and the tile's 64 scale bytes follow its nibbles (layout in k3moe_internal.cuh).
#include "k3moe_internal.cuh"

namespace k3 {
namespace {

constexpr int kWordsPerTile = kTileBytes / 4;  // 272: 256 nibble words + 16 scale words

__global__ void pack_kernel(const uint8_t* __restrict__ canon_nib, const uint8_t* __restrict__ canon_scl,
                            int n_exp, int d, int f, uint8_t* __restrict__ dst, int32_t* bad) {
  const int kt_gu = d / kTileCols, kt_dn = f / kTileCols;
  const long long tiles_gu = (long long)(f / kTileRows) * kt_gu * 2;
  const long long tiles_dn = (long long)(d / kTileRows) * kt_dn;
  const long long tiles_exp = tiles_gu + tiles_dn;
  const long long words_exp = tiles_exp * kWordsPerTile;
  const size_t exp_bytes = packed_expert_bytes(d, f);
  const size_t can_nib = 3ull * f * d / 2, can_scl = 3ull * f * d / 32;
  const size_t mat_nib = (size_t)f * d / 2, mat_scl = (size_t)f * d / 32;
  const long long total = words_exp * n_exp;
  uint32_t smin = 255u, smax = 0u;  // range of the scale bytes this thread saw
  for (long long gw = blockIdx.x * (long long)blockDim.x + threadIdx.x; gw < total;
       gw += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(gw / words_exp);
    const long long wexp = gw % words_exp;
    const long long tile = wexp / kWordsPerTile;
    const int wt = (int)(wexp % kWordsPerTile);
    int m, rg, kt, cols;
    if (tile < tiles_gu) {
      m = (int)(tile & 1);
      const long long q = tile >> 1;
      rg = (int)(q / kt_gu);
      kt = (int)(q % kt_gu);
      cols = d;
    } else {
      m = 2;
      const long long q = tile - tiles_gu;
      rg = (int)(q / kt_dn);
      kt = (int)(q % kt_dn);
      cols = f;
    }
    const uint8_t* nib = canon_nib + (size_t)e * can_nib + (size_t)m * mat_nib;
    const uint8_t* scl = canon_scl + (size_t)e * can_scl + (size_t)m * mat_scl;
    const int rowb = rg * kTileRows;
    uint32_t word = 0;
    if (wt < 256) {
      const int u = wt >> 7, lane = (wt >> 2) & 31, s = wt & 3;
      const int g = lane >> 2, t = lane & 3;
      const int kb = kt * kTileCols + 64 * u + 16 * s;
      const size_t rb = (size_t)cols / 2;
      const uint32_t b0 = nib[(size_t)(rowb + g) * rb + (kb + 2 * t) / 2];
      const uint32_t b1 = nib[(size_t)(rowb + g + 8) * rb + (kb + 2 * t) / 2];
      const uint32_t b2 = nib[(size_t)(rowb + g) * rb + (kb + 2 * t + 8) / 2];
      const uint32_t b3 = nib[(size_t)(rowb + g + 8) * rb + (kb + 2 * t + 8) / 2];
      word = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    } else {
      const int ws = wt - 256, g = ws >> 1, h = ws & 1;
      const size_t sb = (size_t)cols / 32;
      const int row = rowb + g + 8 * h;
      for (int b = 0; b < 4; ++b) {
        const uint32_t sv = scl[(size_t)row * sb + kt * 4 + b];
        if (sv == 255u) atomicOr(bad, 1);  // E8M0 NaN: refused
        if (sv == 0u) atomicOr(bad, 2);    // 2^-127: kernels take the exact subnormal path
        smin = min(smin, sv);
        smax = max(smax, sv);
        word |= sv << (8 * b);
      }
    }
    reinterpret_cast<uint32_t*>(dst + (size_t)e * exp_bytes + (size_t)tile * kTileBytes)[wt] = word;
  }
  // bad[1], bad[2]: smallest and largest scale byte of the layer (the tensor-core path needs
  // their span to fit fp16)
  smin = __reduce_min_sync(0xffffffffu, smin);
  smax = __reduce_max_sync(0xffffffffu, smax);
  if ((threadIdx.x & 31) == 0) {
    if (smin != 255u) atomicMin(bad + 1, (int32_t)smin);
    if (smax != 0u) atomicMax(bad + 2, (int32_t)smax);
  }
}

}  // namespace

cudaError_t launch_pack(const uint8_t* canon_nib, const uint8_t* canon_scl, int n_exp, int d, int f, uint8_t* dst,
                        int32_t* bad, cudaStream_t s) {
  pack_kernel<<<148 * 8, 256, 0, s>>>(canon_nib, canon_scl, n_exp, d, f, dst, bad);
  return cudaGetLastError();
}

}  // namespace k3
