// MXFP8 quantization for the FP8 grouped expert GEMM.
//
// Source: xtuner PR "Decouple expert parallelism from FSDP sharding (dp2ep
// layout)", "Changes" (the Float8 bullet: tile-wise scaling) and
// "Verification" (tile-wise FP8 runs); the pages fix no format, so this library
// takes the block-scaled format the GB300 tensor cores read natively (OCP
// Microscaling MXFP8): E4M3 elements, and for every 32 consecutive elements
// along the reduction dimension K one power-of-two scale 2^X stored as an
// 8-bit biased exponent (code X + 127), X = floor(log2(max |v|)) - 8
// (E4M3's largest exponent), clamped to [-127, 127] (an all-zero block takes
// -127); elements are v / 2^X rounded to the nearest E4M3 value, ties to even,
// saturating at 448.
//
// Scale layout (what the GEMM's tcgen05.cp copies into TMEM): 512-byte atoms of
// 128 rows x 4 K32 scales, row r of the atom at byte (r % 32) * 16 +
// (r / 32) * 4 + j for its j-th K32 block of the atom's 128 K. Atoms are
// ordered [row tile][K / 128].
//  * Activations (rows of the dispatched tokens, K contiguous): the row tiles
//    follow the GEMM's tile list, expert by expert: expert e's rows start at
//    tile 2 * P(e), P(e) = sum over earlier experts of ceil(ceil(n / 128) / 2)
//    (the pairs of 128-row m-tiles), so tile 2 mg + rank holds the rows of the
//    pair tile mg's CTA rank. Rows of a tile past its expert's end have no
//    scale written (the GEMM never stores their results).
//  * Weights [E, K, N] (N contiguous): transposed to K-major rows [E, Nq, K] with
//    tiles of 128 rows; gate and up are interleaved in blocks of 128 rows (rows
//    256 t .. +127 gate columns 128 t .. +127, rows 256 t + 128 .. +255 the same
//    up columns), so 256 rows are one pair GEMM's B with its SwiGLU halves.
//
// Both kernels are HBM-bound streams: 16-byte loads of bf16, 8- or 16-byte
// stores of E4M3, a scale byte per 32 elements.
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// Rows of x [M, K] bf16 -> q [M, K] E4M3 and scale atoms (expert-ordered row tiles).
// A CTA takes RPI whole rows at a time (grid-stride) and issues all their loads
// before it converts any; within a row a thread takes 16 consecutive elements
// (two 16-byte loads), the two threads of a pair share a K32 block (amax by one
// shuffle), and the eight threads of a 128-element atom column gather their four
// scale bytes into one 32-bit store (the atom keeps a row's four K32 scales in
// consecutive bytes). A row's expert and scale tile come from a binary search
// over the offsets once per row. Loops advance whole warps, so every lane
// reaches every shuffle.
template <int RPI>
__global__ void __launch_bounds__(kQThreads)
quantize_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ offsets, int E,
                     int M, int K, uint4* __restrict__ q, uint8_t* __restrict__ sf) {
  pdl_enter();
  extern __shared__ int smq[];
  int* s_off = smq;            // [E + 1]
  int* s_tile = smq + E + 1;   // [E + 1]: first scale tile of each expert
  for (int e = threadIdx.x; e <= E; e += kQThreads) s_off[e] = __ldg(offsets + e);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base <= E; base += 32) {
      const int i = base + lane;
      const int v = (i < E) ? 2 * (((s_off[i + 1] - s_off[i] + 127) / 128 + 1) / 2) : 0;
      int y = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += t;
      }
      if (i <= E) s_tile[i] = carry + y - v;
      carry += __shfl_sync(0xffffffffu, y, 31);
    }
  }
  __syncthreads();
  const int nv = K / 16;   // 16-element pieces per row
  const int kq = K / 128;
  const int rows = s_off[E] < M ? s_off[E] : M;
  const int span = ((nv + 31) / 32) * 32;   // whole warps
  for (int r0 = blockIdx.x * RPI; r0 < rows; r0 += gridDim.x * RPI) {
    long long tile[RPI];
    int rr[RPI];
    bool live[RPI];
#pragma unroll
    for (int i = 0; i < RPI; ++i) {
      const int r = r0 + i;
      live[i] = r < rows;
      int lo = 0, hi = E - 1;   // the expert holding row r: largest e with off[e] <= r
      while (live[i] && lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= r) lo = mid; else hi = mid - 1;
      }
      const int local = r - s_off[lo];
      tile[i] = s_tile[lo] + local / 128;
      rr[i] = local & 127;
    }
    for (int v = threadIdx.x; v < span; v += kQThreads) {
      const bool valid = v < nv;
      uint4 a[RPI], b[RPI];
#pragma unroll
      for (int i = 0; i < RPI; ++i) {
        if (valid && live[i]) {
          const uint4* xr = x + static_cast<size_t>(r0 + i) * (K / 8);
          a[i] = ldg_nc_v4(xr + 2 * v);
          b[i] = ldg_nc_v4(xr + 2 * v + 1);
        } else {
          a[i] = b[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int i = 0; i < RPI; ++i) {
        float f[16];
        unpack8(a[i], f);
        unpack8(b[i], f + 8);
        float amax = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) amax = fmaxf(amax, fabsf(f[u]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const int X = mx_exponent(amax);
        const float sc = inv_pow2(X);
        // the K32 block's scale byte (pair leader), gathered over the atom's four blocks
        const uint32_t byte = static_cast<uint32_t>(X + 127) & 0xffu;
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, byte, 2);
        const uint32_t b2 = __shfl_down_sync(0xffffffffu, byte, 4);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, byte, 6);
        if (!valid || !live[i]) continue;
        uint4 o;
        o.x = to_e4m3x4(f[0] * sc, f[1] * sc, f[2] * sc, f[3] * sc);
        o.y = to_e4m3x4(f[4] * sc, f[5] * sc, f[6] * sc, f[7] * sc);
        o.z = to_e4m3x4(f[8] * sc, f[9] * sc, f[10] * sc, f[11] * sc);
        o.w = to_e4m3x4(f[12] * sc, f[13] * sc, f[14] * sc, f[15] * sc);
        q[static_cast<size_t>(r0 + i) * nv + v] = o;
        if ((lane & 7) == 0) {   // v is a multiple of 8: the atom column v / 8
          const long long atom = tile[i] * kq + v / 8;
          *reinterpret_cast<uint32_t*>(sf + atom_byte(atom, rr[i], 0)) =
              byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
      }
    }
  }
}

// Weights w [E, K, N] bf16 (N contiguous; with w_b, gate and up interleaved)
// -> q [E, Nq, K] E4M3 (K contiguous) and scale atoms [E, Nq / 128, K / 128].
// One CTA per (expert, K32 block, 128 output rows); a thread owns one output
// row: it reads its column's 32 K values (a warp reads 64 contiguous bytes per
// K row), scales them and writes 32 contiguous bytes.
__global__ void __launch_bounds__(128)
quantize_weights_kernel(const __nv_bfloat16* __restrict__ wa, const __nv_bfloat16* __restrict__ wb,
                        int K, int N, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  pdl_enter();
  const int Nq = wb ? 2 * N : N;   // with wb: N % 128 == 0, so 2N % 256 == 0
  const int n_tiles = Nq / 128;
  const int kb32 = K / 32;
  long long b = blockIdx.x;
  const int nt = static_cast<int>(b % n_tiles);
  b /= n_tiles;
  const int j = static_cast<int>(b % kb32);
  const int e = static_cast<int>(b / kb32);
  const int t = threadIdx.x;
  const int nrow = nt * 128 + t;
  const __nv_bfloat16* src = wa;
  int col = nrow;
  if (wb) {
    src = ((nrow >> 7) & 1) ? wb : wa;
    col = (nrow >> 8) * 128 + (nrow & 127);
  }
  const __nv_bfloat16* p = src + (static_cast<size_t>(e) * K + static_cast<size_t>(j) * 32) * N + col;
  float v[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __bfloat162float(p[static_cast<size_t>(i) * N]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int X = mx_exponent(amax);
  const float s = inv_pow2(X);
  uint4 o[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = to_e4m3x4(v[4 * i] * s, v[4 * i + 1] * s, v[4 * i + 2] * s, v[4 * i + 3] * s);
  uint4* dst = reinterpret_cast<uint4*>(q + (static_cast<size_t>(e) * Nq + nrow) * K +
                                        static_cast<size_t>(j) * 32);
  dst[0] = o[0];
  dst[1] = o[1];
  const long long atom = (static_cast<long long>(e) * n_tiles + nt) * (K / 128) + j / 4;
  sf[atom_byte(atom, t, j)] = static_cast<uint8_t>(X + 127);
}

}  // namespace

// Scale tiles the activation layout needs for M rows over E experts (an upper
// bound of 2 * sum_e ceil(ceil(n_e / 128) / 2)).
long long mxfp8_row_tiles(long long M, int E) { return (M + 127) / 128 + 2LL * E; }

int launch_quantize_rows(const void* x, const int32_t* offsets, int E, int M, int K, void* q,
                         void* sf, cudaStream_t st) {
#ifndef MOE_QROWS_RPI
#define MOE_QROWS_RPI 2
#endif
  constexpr int kRpi = MOE_QROWS_RPI;   // rows per CTA iteration
  long long grid = (M + kRpi - 1) / kRpi;   // at most eight resident CTAs per SM (grid-stride)
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const size_t smem = sizeof(int) * 2 * (E + 1);
  ProfScope prof("mxfp8_quantize_rows", st);
  return launch_pdl(quantize_rows_kernel<kRpi>, static_cast<unsigned>(grid), kQThreads, smem, st, 1,
                    static_cast<const uint4*>(x), offsets, E, M, K, static_cast<uint4*>(q),
                    static_cast<uint8_t*>(sf));
}

}  // namespace moe

extern "C" int moe_mxfp8_quantize_rows(const moe_bf16* x, const int32_t* offsets, int E, int M,
                                       int K, uint8_t* q, uint8_t* sf, void* stream) {
  using namespace moe;
  if (E < 1 || E > 1024 || M < 0 || K <= 0 || K % 128) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!x || !offsets || !q || !sf) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(offsets) || !aligned16(q) || !aligned16(sf))
    return MOE_ERR_MISALIGNED;
  return launch_quantize_rows(x, offsets, E, M, K, q, sf, as_stream(stream));
}

extern "C" int moe_mxfp8_quantize_weights(const moe_bf16* w_a, const moe_bf16* w_b, int E, int K,
                                          int N, uint8_t* q, uint8_t* sf, void* stream) {
  using namespace moe;
  if (E < 1 || K <= 0 || N <= 0 || K % 128 || N % 128) return MOE_ERR_INVALID_ARG;
  if (!w_a || !q || !sf) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w_a) || (w_b && !aligned16(w_b)) || !aligned16(q) || !aligned16(sf))
    return MOE_ERR_MISALIGNED;
  const int Nq = w_b ? 2 * N : N;
  const long long blocks = static_cast<long long>(E) * (K / 32) * (Nq / 128);
  if (blocks > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = as_stream(stream);
  ProfScope prof("mxfp8_quantize_weights", st);
  return launch_pdl(quantize_weights_kernel, static_cast<unsigned>(blocks), 128, 0, st, 1,
                    reinterpret_cast<const __nv_bfloat16*>(w_a),
                    reinterpret_cast<const __nv_bfloat16*>(w_b), K, N, q, static_cast<uint8_t*>(sf));
}

namespace moe {
MOE_DEBUG_STATUS_READER(fp8)
}  // namespace moe
