// Grouped expert GEMMs on the CUDA cores (FFMA, float32 accumulation).
//
// This is the strict-float32 path of the layer (no TF32 rounding of the
// operands), and it serves every contraction of the forward and the train
// step:
//   LOGITS  logits = x W_r
//   GU      a_g = x_t W_gate[e], a_u = x_t W_up[e], H = silu(a_g) * a_u
//           (gather of the token rows fused into the operand load)
//   DOWN    gate * (H W_down[e]) per sorted row (the pair's share of y[t])
//   DZ      Z = dy_t W_down[e]^T; gate * dgate = gate * <Z, H> (the router
//           backward's q); dA_g, dA_u by the SwiGLU chain rule; gH = gate * H
//           kept for the W_down gradient
//   DX      dA_g W_gate[e]^T + dA_u W_up[e]^T per sorted row (share of dx[t])
//   DWD     dW_down[e] = sum_r gH_r^T dy_t           (ragged K = expert rows)
//   DWGU    dW_gate[e] | dW_up[e] = sum_r x_t^T [dA_g | dA_u]
// Each kind also runs densely (one expert, identity row map) for the shared
// expert.  The method these follow: the experts_grouped_swiglu and
// unpermute_combine pieces of kernel_gmm_gpu.json and the value_and_grad
// train step of gpu_moe_h100.json.
#include <cmath>

#include "kernels.cuh"

namespace moe {
namespace {

enum Kind { LOGITS, GU, DOWN, DZ, DX, DWD, DWGU };

constexpr int BK = 16, NT = 256;

// The tile edge of a GEMM whose output has N columns and (weight
// gradients) M rows: 128 where both divide, else 64.
inline int tile_of(int64_t N, int64_t M = 128) { return N % 128 == 0 && M % 128 == 0 ? 128 : 64; }
// Columns of W_gate (and of W_up) per gate/up tile of `tm` rows.
inline int gu_cols(int tm) { return tm == 128 ? 64 : tm; }

struct SimtArgs {
  // operands
  const void* A = nullptr;
  const void* B = nullptr;
  const void* B2 = nullptr;  // GU: W_up; DX: W_up (second half of K)
  int lda = 0, ldb = 0;
  int64_t b_estride = 0;     // elements between consecutive experts' B matrices
  int N = 0, K = 0;          // output columns; reduction length of the row GEMMs
  int64_t rows = 0;          // dense kinds: number of rows
  int h = 0;                 // DX: K split point; DWGU: N split point; DZ: hidden width
  // dispatch tables
  const int4* tiles = nullptr;
  const int* ntiles = nullptr;
  const int32_t* rowpair = nullptr;
  int top_k = 1;
  const int* counts = nullptr;
  const int* poff = nullptr;
  const float* gates = nullptr;
  // epilogue operands / outputs
  void* h_out = nullptr;         // GU
  void* ag_out = nullptr;        // GU (train)
  void* au_out = nullptr;        // GU (train)
  const void* ag_in = nullptr;   // DZ
  const void* au_in = nullptr;   // DZ
  void* dA_out = nullptr;        // DZ  [rows, 2h]
  void* gH_out = nullptr;        // DZ  [rows, h]
  float* dg_part = nullptr;      // DZ  [rows, dg_ld]
  int dg_ld = 0;
  void* slot_out = nullptr;      // DOWN / DX: one row per sorted (or dense) row
  float* acc_out = nullptr;      // LOGITS / DWD / DWGU (gate half)
  const float* col_bias = nullptr;  // LOGITS: router bias [N], nullable
  float* acc_out2 = nullptr;     // DWGU (up half)
  int ldo = 0;
  int n_ntiles = 1, n_mtiles = 1;
  int tm = 64;                   // tile edge: 64, or 128 where the dimensions divide
  // DW kinds: each expert's K range cut into ksplit chunks of whole K steps
  // (more blocks, so that the last wave of tiles is nearly full); chunk s
  // writes its partial tile to part + s * part_sstride, rows e * M + m, row
  // stride n_ntiles * TM, summed afterwards in chunk order
  int ksplit = 1;
  float* part = nullptr;
  int64_t part_sstride = 0;
};

template <typename T>
__device__ __forceinline__ float4 load4(const T* p, bool ok) {
  if (!ok) return make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (sizeof(T) == 4) {
    return *reinterpret_cast<const float4*>(p);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
  }
}

template <typename T>
__device__ __forceinline__ float load1(const T* p, bool ok) {
  return ok ? to_f32(*p) : 0.f;
}

// four consecutive elements (16 bytes of float, 8 of bf16; 4-element aligned)
template <typename T>
__device__ __forceinline__ void store4(T* p, float a, float b, float c, float d) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
  }
}

__device__ __forceinline__ float comp(const float4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// TM x TM output tiles (TM = 64 or 128), 256 threads as 16 x 16, each
// thread an R x R micro-tile (R = TM / 16: 4 or 8) made of (R / 4)^2 blocks
// of 4 x 4 elements 64 rows / columns apart (its rows ty*4 + i + 64*u, its
// columns tx*4 + j + 64*v), so that every shared-memory operand read is a
// conflict-free float4 and the 16 threads of a row are 16 consecutive lanes.
// The 8 x 8 micro-tile issues 64 FFMAs per 4 float4 loads of each k step,
// the 4 x 4 one 16 per 2.  The gate/up projection's 128-row tiles are 64
// columns wide in each of its two weights (8 x 4 micro-tiles, two of them).
template <Kind KIND, typename T, bool ROUTED, int TM>
__device__ __forceinline__ void simt_gemm_body(const SimtArgs& a) {
  constexpr bool A_KCONTIG = (KIND == LOGITS || KIND == GU || KIND == DOWN || KIND == DZ ||
                              KIND == DX);
  constexpr bool B_KCONTIG = (KIND == DZ || KIND == DX);
  constexpr bool DUAL = (KIND == GU);
  constexpr bool DW = (KIND == DWD || KIND == DWGU);
  constexpr int R = TM / 16;   // micro-tile edge
  constexpr int U = TM / 64;   // 4 x 4 blocks per micro-tile edge; loads per thread per operand
  // the tile's column extent: the gate/up projection's 128-row tiles take 64
  // columns of each of its two weight matrices (two 8 x 4 accumulator sets
  // per thread, so that two blocks fit an SM); every other tile is square
  constexpr int TN = DUAL && TM == 128 ? 64 : TM;
  constexpr int RN = TN / 16, UN = TN / 64;  // micro-tile columns; B loads per thread

  // the operand tiles in dynamic shared memory; the weight-gradient and dZ
  // kinds keep two buffers of each (the next K step's tile is stored into
  // one while the other is read: one barrier per K step), the others one
  // (measured faster for them)
  constexpr int NB = (KIND == DWD || KIND == DWGU || KIND == DZ) ? 2 : 1;
  typedef float Tile_[BK][TM + 4];
  // one buffer: static arrays (fixed addresses); two: dynamic shared memory
  constexpr int SR = NB == 1 ? BK : 1, SC = NB == 1 ? TM + 4 : 4;
  __shared__ __align__(16) float As1[SR][SC];
  __shared__ __align__(16) float Bs1[SR][SC];
  __shared__ __align__(16) float Bs21[DUAL && NB == 1 ? BK : 1][DUAL && NB == 1 ? TM + 4 : 4];
  extern __shared__ __align__(16) float simt_smem[];
  Tile_* As = NB == 1 ? reinterpret_cast<Tile_*>(&As1[0][0]) : reinterpret_cast<Tile_*>(simt_smem);
  Tile_* Bs = NB == 1 ? reinterpret_cast<Tile_*>(&Bs1[0][0]) : As + NB;
  Tile_* Bs2 = NB == 1 ? reinterpret_cast<Tile_*>(&Bs21[0][0]) : Bs + NB;  // DUAL only
  __shared__ int s_tok[TM];  // source rows of the tile (row kinds)
  // routed down projection: each row's gate, read once before the main loop
  // instead of by dependent loads in the epilogue (measured 5.00 -> 4.83 ms
  // at E8/k2, 131072 tokens; the same for dZ measured slower, 6.48 -> 7.01)
  constexpr bool ROWGATE = ROUTED && KIND == DOWN;
  __shared__ float s_gt[ROWGATE ? TM : 1];

  const int tid = threadIdx.x;
  const int ntile = blockIdx.x % a.n_ntiles;
  const int rest = blockIdx.x / a.n_ntiles;
  const int n0 = ntile * TN;

  int e = 0;
  int64_t row0 = 0;     // first output row (row kinds) / first K row (DW kinds)
  int nvalid = 0;       // row kinds: valid rows in this tile
  int m0 = 0;           // DW kinds: first output row
  int chunk = 0;        // DW kinds: chunk of the expert's K range
  int64_t kbeg = 0, kend = 0;

  if constexpr (!DW) {
    if constexpr (ROUTED) {
      // tile-list entries hold 128 rows: one block (TM = 128) or two halves
      constexpr int PER = 128 / TM;
      const int mt = rest / PER, part = rest % PER;
      if (mt >= a.ntiles[0]) return;
      const int4 tile = a.tiles[mt];
      e = tile.x;
      row0 = tile.y + part * TM;
      nvalid = min(TM, tile.z - part * TM);
      if (nvalid <= 0) return;
    } else {
      row0 = (int64_t)rest * TM;
      if (row0 >= a.rows) return;
      nvalid = a.rows - row0 < TM ? (int)(a.rows - row0) : TM;
    }
    for (int i = tid; i < TM; i += NT) {
      int64_t src = row0 + i;
      if constexpr (ROUTED) {
        if (KIND == GU || KIND == DZ || ROWGATE) {
          const int32_t p = i < nvalid ? a.rowpair[row0 + i] : -1;
          if (KIND != DOWN) src = p >= 0 ? p / a.top_k : 0;
          if constexpr (ROWGATE) s_gt[i] = p >= 0 ? __ldg(a.gates + p) : 0.f;
        }
      }
      s_tok[i] = (int)src;  // token (gathered kinds) or sorted row
    }
    kbeg = 0;
    kend = a.K;
  } else {
    // blocks in the order (expert, chunk, row tile, column tile): the
    // blocks that run together read the same K rows
    const int mt = rest % a.n_mtiles;
    const int es = rest / a.n_mtiles;
    e = es / a.ksplit;
    chunk = es % a.ksplit;
    m0 = mt * TM;
    int64_t k0, n;
    if constexpr (ROUTED) {
      k0 = a.poff[e];
      n = a.counts[e];
    } else {
      k0 = 0;
      n = a.rows;
    }
    const int64_t steps = (n + BK - 1) / BK;
    kbeg = k0 + BK * (steps * chunk / a.ksplit);
    kend = k0 + BK * (steps * (chunk + 1) / a.ksplit);
    if (kend > k0 + n) kend = k0 + n;
    if (kend < kbeg) kend = kbeg;
  }
  __syncthreads();

  const T* A = reinterpret_cast<const T*>(a.A);
  const T* B = reinterpret_cast<const T*>(a.B) + (ROUTED ? a.b_estride * e : 0);
  const T* B2 = a.B2 ? reinterpret_cast<const T*>(a.B2) + (ROUTED ? a.b_estride * e : 0) : nullptr;

  float acc[R][RN] = {};
  float acc2[DUAL ? R : 1][DUAL ? RN : 1] = {};
  const int ty = tid / 16, tx = tid % 16;

  // routed DW kinds gather token rows along K: this thread's K row (the same
  // for A and B) maps to its token through rowpair, read one K step before
  // the operand loads that use it
  constexpr bool GATHER_K = DW && ROUTED;
  int64_t ktok = 0;      // token row of the step being loaded
  int32_t pair_next = 0; // rowpair entry of the step after it
  auto kpair = [&](int64_t kt) -> int32_t {
    const int64_t r = kbeg + kt + tid / 16;
    return r < kend ? __ldg(a.rowpair + r) : 0;
  };
  float4 ra[U], rb[UN], rb2[DUAL ? UN : 1];
  auto gload = [&](int64_t kt) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      // ---- A ----
      if constexpr (A_KCONTIG) {
        const int m = tid / 4 + 64 * u, k4 = (tid % 4) * 4;
        const bool ok = m < nvalid || (KIND == DOWN || KIND == DX);
        const int64_t src = (KIND == LOGITS || !ROUTED) ? row0 + m : (int64_t)s_tok[m];
        const bool in = ok && (ROUTED || row0 + m < a.rows);
        ra[u] = load4(A + src * a.lda + kt + k4, in);
      } else {
        const int kl = tid / 16, m4 = (tid % 16) * 4 + 64 * u;
        const int64_t r = kbeg + kt + kl;
        const bool ok = r < kend;
        const int64_t src = KIND == DWGU && ROUTED ? ktok : r;
        ra[u] = load4(A + src * a.lda + m0 + m4, ok);
      }
      // ---- B ----
      if (u >= UN) continue;
      if constexpr (!B_KCONTIG) {
        const int kl = tid / 16, n4 = (tid % 16) * 4 + 64 * u;
        if constexpr (KIND == LOGITS) {
          const int64_t kk = kt + kl;
          float v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = load1(B + kk * a.ldb + n0 + n4 + q, n0 + n4 + q < a.N);
          rb[u] = make_float4(v[0], v[1], v[2], v[3]);
        } else if constexpr (DW) {
          const int64_t r = kbeg + kt + kl;
          const bool ok = r < kend;
          const int64_t src = KIND == DWD && ROUTED ? ktok : r;
          rb[u] = load4(B + src * a.ldb + n0 + n4, ok);
        } else {
          const int64_t kk = kt + kl;
          rb[u] = load4(B + kk * a.ldb + n0 + n4, true);
          if constexpr (DUAL) rb2[u] = load4(B2 + kk * a.ldb + n0 + n4, true);
        }
      } else {
        const int n = tid / 4 + 64 * u, k4 = (tid % 4) * 4;
        const int64_t kk = kt + k4;
        if constexpr (KIND == DX) {
          const T* src = kk < a.h ? B + (int64_t)(n0 + n) * a.ldb + kk
                                  : B2 + (int64_t)(n0 + n) * a.ldb + (kk - a.h);
          rb[u] = load4(src, true);
        } else {
          rb[u] = load4(B + (int64_t)(n0 + n) * a.ldb + kk, true);
        }
      }
    }
  };
  auto sstore = [&](int buf) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if constexpr (A_KCONTIG) {
        const int m = tid / 4 + 64 * u, k4 = (tid % 4) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) As[buf][k4 + q][m] = comp(ra[u], q);
      } else {
        const int kl = tid / 16, m4 = (tid % 16) * 4 + 64 * u;
        *reinterpret_cast<float4*>(&As[buf][kl][m4]) = ra[u];
      }
      if (u >= UN) continue;
      if constexpr (!B_KCONTIG) {
        const int kl = tid / 16, n4 = (tid % 16) * 4 + 64 * u;
        *reinterpret_cast<float4*>(&Bs[buf][kl][n4]) = rb[u];
        if constexpr (DUAL) *reinterpret_cast<float4*>(&Bs2[buf][kl][n4]) = rb2[u];
      } else {
        const int n = tid / 4 + 64 * u, k4 = (tid % 4) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) Bs[buf][k4 + q][n] = comp(rb[u], q);
      }
    }
  };

  const int64_t klen = kend - kbeg;
  int cur = 0;
  if constexpr (GATHER_K) {
    if (klen > 0) {
      ktok = kpair(0) / a.top_k;
      pair_next = kpair(BK);
    }
  }
  if constexpr (NB == 2) {
    if (klen > 0) {
      gload(0);
      sstore(0);
    }
    __syncthreads();
  } else {
    if (klen > 0) gload(0);
  }
  for (int64_t kt = 0; kt < klen; kt += BK) {
    // the next K step's operands: global loads now, their shared-memory
    // stores after this step's FMAs (two buffers) or before them (one)
    const bool more = kt + BK < klen;
    if constexpr (NB == 1) {
      __syncthreads();
      sstore(0);
      __syncthreads();
    }
    if (more) {
      if constexpr (GATHER_K) {
        ktok = pair_next / a.top_k;
        pair_next = kpair(kt + 2 * BK);
      }
      gload(kt + BK);
    }
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float am[R], bn[RN], bn2[DUAL ? RN : 1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float4 av = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4 + 64 * u]);
        am[4 * u] = av.x; am[4 * u + 1] = av.y; am[4 * u + 2] = av.z; am[4 * u + 3] = av.w;
        if (u >= UN) continue;
        const float4 bv = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4 + 64 * u]);
        bn[4 * u] = bv.x; bn[4 * u + 1] = bv.y; bn[4 * u + 2] = bv.z; bn[4 * u + 3] = bv.w;
        if constexpr (DUAL) {
          const float4 b2 = *reinterpret_cast<const float4*>(&Bs2[cur][kk][tx * 4 + 64 * u]);
          bn2[4 * u] = b2.x; bn2[4 * u + 1] = b2.y; bn2[4 * u + 2] = b2.z; bn2[4 * u + 3] = b2.w;
        }
      }
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(am[i], bn[j], acc[i][j]);
      if constexpr (DUAL) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int j = 0; j < RN; ++j) acc2[i][j] = fmaf(am[i], bn2[j], acc2[i][j]);
      }
    }
    if constexpr (NB == 2) {
      if (more) sstore(cur ^ 1);
      __syncthreads();  // the other buffer is full; every thread has left this one
      cur ^= 1;
    }
  }

  // ---------------- epilogues ----------------
  // micro-tile element (i, j): row ty*4 + (i % 4) + 64*(i / 4), column
  // tx*4 + (j % 4) + 64*(j / 4) of the tile; the four columns of a j block
  // are consecutive and move as one vector
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int m = ty * 4 + (i & 3) + 64 * (i >> 2);
    const int64_t r = row0 + m;
    if constexpr (KIND == LOGITS) {
      if (r < a.rows)
#pragma unroll
        for (int j = 0; j < RN; ++j) {
          const int n = n0 + tx * 4 + (j & 3) + 64 * (j >> 2);
          if (n < a.N) a.acc_out[r * a.ldo + n] = acc[i][j] + (a.col_bias ? a.col_bias[n] : 0.f);
        }
    } else if constexpr (KIND == GU) {
      if (!ROUTED && r >= a.rows) continue;
      T* H = reinterpret_cast<T*>(a.h_out);
      T* AG = reinterpret_cast<T*>(a.ag_out);
      T* AU = reinterpret_cast<T*>(a.au_out);
#pragma unroll
      for (int jb = 0; jb < UN; ++jb) {
        const int64_t o = r * a.ldo + n0 + tx * 4 + 64 * jb;
        // round to the storage type first, so H is computed from exactly the
        // values a backward pass reads back
        float g[4], u[4], hv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          g[c] = to_f32(from_f32<T>(acc[i][4 * jb + c]));
          u[c] = to_f32(from_f32<T>(acc2[i][4 * jb + c]));
          hv[c] = g[c] * sigmoidf_(g[c]) * u[c];
        }
        store4(H + o, hv[0], hv[1], hv[2], hv[3]);
        if (AG) {
          store4(AG + o, g[0], g[1], g[2], g[3]);
          store4(AU + o, u[0], u[1], u[2], u[3]);
        }
      }
    } else if constexpr (KIND == DOWN || KIND == DX) {
      // one output row per sorted row (routed: the pair's share of its
      // token's output, gate applied for DOWN; dense: the shared expert's
      // row); the combine gathers the shares of a token in a fixed order
      if (m >= nvalid) continue;
      float sc = 1.f;
      if constexpr (ROUTED && KIND == DOWN) sc = s_gt[m];
      T* out = reinterpret_cast<T*>(a.slot_out);
#pragma unroll
      for (int j = 0; j < RN; ++j)
        out[r * a.ldo + n0 + tx * 4 + (j & 3) + 64 * (j >> 2)] = from_f32<T>(sc * acc[i][j]);
    } else if constexpr (KIND == DZ) {
      const bool exists = ROUTED || r < a.rows;
      const bool valid = m < nvalid;
      float gt = 1.f;
      if constexpr (ROUTED) gt = valid ? a.gates[a.rowpair[r]] : 0.f;
      const T* AG = reinterpret_cast<const T*>(a.ag_in);
      const T* AU = reinterpret_cast<const T*>(a.au_in);
      T* dA = reinterpret_cast<T*>(a.dA_out);
      T* gH = reinterpret_cast<T*>(a.gH_out);
      const int64_t h = a.h;
      float dgp = 0.f;
#pragma unroll
      for (int j = 0; j < RN; ++j) {
        const int n = n0 + tx * 4 + (j & 3) + 64 * (j >> 2);
        const float z = acc[i][j];
        const float ag = valid ? to_f32(AG[r * h + n]) : 0.f;
        const float au = valid ? to_f32(AU[r * h + n]) : 0.f;
        const float s = sigmoidf_(ag);
        const float sl = ag * s;
        const float hv = to_f32(from_f32<T>(sl * au));  // H as the forward stored it
        dgp += z * hv;
        const float dh = gt * z;
        const float dau = dh * sl;
        const float dag = dh * au * s * (1.f + ag * (1.f - s));
        if (exists) {
          dA[r * 2 * h + n] = from_f32<T>(valid ? dag : 0.f);
          dA[r * 2 * h + h + n] = from_f32<T>(valid ? dau : 0.f);
          gH[r * h + n] = from_f32<T>(valid ? gt * hv : 0.f);
        }
      }
      // the 16 threads of one row are 16 consecutive lanes of a warp
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) dgp += __shfl_xor_sync(0xffffffffu, dgp, o);
      if (ROUTED && tx == 0 && valid)
        a.dg_part[(int64_t)a.rowpair[r] * a.dg_ld + ntile] = gt * dgp;
    } else {  // DWD / DWGU: the expert's gradient tile, or a K chunk's partial of it
      const int64_t om = m0 + m;
      const int64_t eoff = (int64_t)e * a.n_mtiles * TM;  // expert offset in rows
#pragma unroll
      for (int jb = 0; jb < UN; ++jb) {
        const int n = n0 + tx * 4 + 64 * jb;
        float* dst;
        if (a.ksplit > 1) {
          dst = a.part + chunk * a.part_sstride + (eoff + om) * ((int64_t)a.n_ntiles * TN) + n;
        } else if constexpr (KIND == DWGU) {
          // a 4-column block never straddles the gate | up boundary (h % 4 == 0)
          dst = n < a.h ? a.acc_out + (eoff + om) * a.h + n
                        : a.acc_out2 + (eoff + om) * a.h + (n - a.h);
        } else {
          dst = a.acc_out + (eoff + om) * a.ldo + n;
        }
        *reinterpret_cast<float4*>(dst) = make_float4(acc[i][4 * jb], acc[i][4 * jb + 1],
                                                      acc[i][4 * jb + 2], acc[i][4 * jb + 3]);
      }
    }
  }
}

// The kernels: the weight-gradient kinds, dX and the 128-row gate/up tiles
// are compiled for two resident 128-row blocks (four 64-row) per SM, at most
// 128 / 64 registers a thread (measured 0.63 -> 0.68 of the FFMA rate for
// dX at 131072 tokens); the other kinds take the registers the compiler
// gives them (the routed down projection and dZ fit two blocks as they are;
// the dense down projection spills under the bound).
template <Kind KIND, typename T, bool ROUTED, int TM>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(const SimtArgs a) {
  simt_gemm_body<KIND, T, ROUTED, TM>(a);
}
template <Kind KIND, typename T, bool ROUTED, int TM>
__global__ void __launch_bounds__(NT, TM == 64 ? 4 : 2) simt_gemm2_kernel(const SimtArgs a) {
  simt_gemm_body<KIND, T, ROUTED, TM>(a);
}
template <Kind KIND, typename T, bool ROUTED, int TM>
constexpr auto simt_kernel() {
  if constexpr (KIND == DWD || KIND == DWGU || KIND == DX || (KIND == GU && TM == 128))
    return simt_gemm2_kernel<KIND, T, ROUTED, TM>;
  else return simt_gemm_kernel<KIND, T, ROUTED, TM>;
}

// Dynamic shared memory of a kernel instance: the two buffers of A and B of
// the double-buffered kinds (the others keep static tiles).
template <Kind KIND, int TM>
constexpr size_t simt_smem_bytes() {
  return (KIND == DWD || KIND == DWGU || KIND == DZ) ? sizeof(float) * BK * (TM + 4) * 2 * 2 : 0;
}

template <Kind KIND, typename T, bool ROUTED, int TM>
void launch_tm(const SimtArgs& a, int64_t blocks, const char* name, cudaStream_t s) {
  constexpr size_t smem = simt_smem_bytes<KIND, TM>();
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(simt_kernel<KIND, T, ROUTED, TM>(),
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  MOE_LAUNCH(name, s, simt_kernel<KIND, T, ROUTED, TM>()<<<(unsigned)blocks, NT, smem, s>>>(a));
}

// Blocks of a kernel instance resident on one SM times the device's SMs
// (the device's, not the launch limit's: the K chunks a weight gradient is
// cut into, and so its summation order, depend on this number alone).
template <Kind KIND, typename T, bool ROUTED, int TM>
int64_t resident_slots() {
  static int64_t slots = 0;
  if (!slots) {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, simt_kernel<KIND, T, ROUTED, TM>(), NT,
                                                  simt_smem_bytes<KIND, TM>());
    slots = (int64_t)(sms > 0 ? sms : 1) * (per > 0 ? per : 1);
  }
  return slots;
}

// K chunks for a weight-gradient GEMM of `tiles` output tiles whose experts
// hold about `krows` rows each: the count (<= kSimtMaxSplit, chunks of at
// least 256 rows, tiles x chunks <= kSimtChunkTiles, the partials' room)
// whose blocks fill their last wave of `slots` best; more chunks only where
// that gains at least 2 % (each adds a partial tile).
inline int dw_chunks(int64_t tiles, int64_t krows, int64_t slots) {
  auto fill = [&](int c) {
    const double w = (double)(tiles * c) / (double)slots;
    return w / std::ceil(w);
  };
  int best = 1;
  double best_fill = fill(1);
  for (int c = 2; c <= kSimtMaxSplit && krows / c >= 256 && tiles * c <= kSimtChunkTiles; ++c) {
    const double f = fill(c);
    if (f > best_fill + 0.02) {
      best = c;
      best_fill = f;
    }
  }
  return best;
}

template <Kind KIND, typename T, bool ROUTED>
void launch(const SimtArgs& a, int64_t blocks, cudaStream_t s) {
  if (blocks <= 0) return;
  static const char* names[2][7] = {
      {"simt_logits", "simt_gateup_sh", "simt_down_sh", "simt_dz_sh", "simt_dx_sh",
       "simt_dw_down_sh", "simt_dw_gateup_sh"},
      {"simt_logits", "simt_gateup", "simt_down", "simt_dz", "simt_dx", "simt_dw_down",
       "simt_dw_gateup"}};
  if (a.tm == 128)
    launch_tm<KIND, T, ROUTED, 128>(a, blocks, names[ROUTED ? 1 : 0][KIND], s);
  else
    launch_tm<KIND, T, ROUTED, 64>(a, blocks, names[ROUTED ? 1 : 0][KIND], s);
}

// A weight-gradient GEMM (DWD / DWGU) of `tiles` output tiles over
// experts of about `krows` rows: cut into K chunks where that fills the
// GPU's last wave better, the chunks' partial tiles (in `part`, room for
// kSimtMaxSplit of them) then summed in chunk order into the outputs.
template <Kind KIND, typename T, bool ROUTED>
void launch_dw(SimtArgs a, int64_t tiles, int64_t krows, float* part, cudaStream_t s) {
  if (tiles <= 0) return;
  const int64_t slots = a.tm == 128 ? resident_slots<KIND, T, ROUTED, 128>()
                                    : resident_slots<KIND, T, ROUTED, 64>();
  // the workspace holds chunk partials for float32 layers (the bf16 layer's
  // weight gradients run on the tensor cores)
  const int c = sizeof(T) == 4 ? dw_chunks(tiles, krows, slots) : 1;
  const int64_t M = (int64_t)a.n_mtiles * a.tm, N = (int64_t)a.n_ntiles * a.tm;
  const int64_t EM = tiles / ((int64_t)a.n_mtiles * a.n_ntiles) * M;
  if (c > 1) {
    a.ksplit = c;
    a.part = part;
    a.part_sstride = EM * N;
  }
  launch<KIND, T, ROUTED>(a, tiles * c, s);
  if (c > 1)
    launch_split_reduce(part, c, EM, (int)N, (int)N, KIND == DWGU ? a.h : 0, a.acc_out,
                        KIND == DWGU ? a.acc_out2 : nullptr, s);
}

template <typename T>
void router_logits_t(const moe_dims& d, const LayerPtrs& p, float* logits, cudaStream_t s) {
  SimtArgs a;
  a.A = p.x;
  a.lda = d.d_model;
  a.B = p.w_router;
  a.ldb = d.experts;
  a.N = d.experts;
  a.K = d.d_model;
  a.rows = d.tokens;
  a.acc_out = logits;
  a.col_bias = p.router_bias;
  a.ldo = d.experts;
  a.n_ntiles = (d.experts + 63) / 64;
  launch<LOGITS, T, false>(a, a.n_ntiles * ((d.tokens + 63) / 64), s);
}

template <typename T>
void grouped_fwd_t(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                   cudaStream_t s) {
  const int h = d.d_hidden, dm = d.d_model;
  SimtArgs a;
  a.tiles = at<int4>(ws, L.tiles);
  a.ntiles = at<int>(ws, L.ntiles);
  a.rowpair = at<int32_t>(ws, L.rowpair);
  a.top_k = d.top_k;
  a.gates = p.gates;
  // gate/up projection with the SwiGLU epilogue
  a.A = p.x;
  a.lda = dm;
  a.B = p.w_gate;
  a.B2 = p.w_up;
  a.ldb = h;
  a.b_estride = (int64_t)dm * h;
  a.N = h;
  a.K = dm;
  a.h_out = p.h_buf;
  a.ag_out = mode == MOE_SAVE_FOR_BWD ? p.a_gate : nullptr;
  a.au_out = mode == MOE_SAVE_FOR_BWD ? p.a_up : nullptr;
  a.ldo = h;
  a.tm = tile_of(h);
  a.n_ntiles = h / gu_cols(a.tm);
  launch<GU, T, true>(a, a.n_ntiles * (128 / a.tm) * L.MTcap, s);
  // down projection with the gate-weighted combine
  SimtArgs b = a;
  b.A = p.h_buf;
  b.lda = h;
  b.B = p.w_down;
  b.B2 = nullptr;
  b.ldb = dm;
  b.b_estride = (int64_t)h * dm;
  b.N = dm;
  b.K = h;
  b.slot_out = at<void>(ws, L.osort);
  b.ldo = dm;
  b.tm = tile_of(dm);
  b.n_ntiles = dm / b.tm;
  launch<DOWN, T, true>(b, b.n_ntiles * (128 / b.tm) * L.MTcap, s);
}

template <typename T>
void shared_fwd_t(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                  cudaStream_t s) {
  const int hs = d.shared_hidden, dm = d.d_model;
  SimtArgs a;
  a.rows = d.tokens;
  a.A = p.x;
  a.lda = dm;
  a.B = p.ws_gate;
  a.B2 = p.ws_up;
  a.ldb = hs;
  a.N = hs;
  a.K = dm;
  a.h_out = p.hs_buf;
  a.ag_out = mode == MOE_SAVE_FOR_BWD ? p.as_gate : nullptr;
  a.au_out = mode == MOE_SAVE_FOR_BWD ? p.as_up : nullptr;
  a.ldo = hs;
  a.tm = tile_of(hs);
  a.n_ntiles = hs / gu_cols(a.tm);
  launch<GU, T, false>(a, a.n_ntiles * ((d.tokens + a.tm - 1) / a.tm), s);
  SimtArgs b = a;
  b.A = p.hs_buf;
  b.lda = hs;
  b.B = p.ws_down;
  b.B2 = nullptr;
  b.ldb = dm;
  b.N = dm;
  b.K = hs;
  b.slot_out = at<void>(ws, L.ys);
  b.ldo = dm;
  b.tm = tile_of(dm);
  b.n_ntiles = dm / b.tm;
  launch<DOWN, T, false>(b, b.n_ntiles * ((d.tokens + b.tm - 1) / b.tm), s);
}

// the shared expert's backward (dxs and its weight gradients)
template <typename T>
void backward_shared_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                       cudaStream_t s) {
  const int dm = d.d_model, hs = d.shared_hidden;
  auto row_tiles = [&](int tm) { return (d.tokens + tm - 1) / tm; };
  if (hs > 0) {
    void* dAs = at<void>(ws, L.dAs);
    void* gHs = at<void>(ws, L.gHs);
    // Z_s = dy Ws_down^T with the SwiGLU chain rule (gate = 1)
    SimtArgs z;
    z.rows = d.tokens;
    z.A = p.dy;
    z.lda = dm;
    z.B = p.ws_down;
    z.ldb = dm;
    z.N = hs;
    z.K = dm;
    z.h = hs;
    z.ag_in = p.as_gate;
    z.au_in = p.as_up;
    z.dA_out = dAs;
    z.gH_out = gHs;
    z.tm = tile_of(hs);
    z.n_ntiles = hs / z.tm;
    launch<DZ, T, false>(z, z.n_ntiles * row_tiles(z.tm), s);
    // dx_acc = dAs [Ws_gate | Ws_up]^T   (plain store: first writer)
    SimtArgs x;
    x.rows = d.tokens;
    x.A = dAs;
    x.lda = 2 * hs;
    x.B = p.ws_gate;
    x.B2 = p.ws_up;
    x.ldb = hs;
    x.N = dm;
    x.K = 2 * hs;
    x.h = hs;
    x.slot_out = at<void>(ws, L.dxs);
    x.ldo = dm;
    x.tm = tile_of(dm);
    x.n_ntiles = dm / x.tm;
    launch<DX, T, false>(x, x.n_ntiles * row_tiles(x.tm), s);
    // dWs_down = Hs^T dy ; dWs_gate | dWs_up = x^T dAs
    SimtArgs w;
    w.rows = d.tokens;
    w.A = gHs;
    w.lda = hs;
    w.B = p.dy;
    w.ldb = dm;
    w.acc_out = p.dws_down;
    w.ldo = dm;
    w.tm = tile_of(dm, hs);
    w.n_mtiles = hs / w.tm;
    w.n_ntiles = dm / w.tm;
    launch_dw<DWD, T, false>(w, (int64_t)w.n_ntiles * w.n_mtiles, d.tokens,
                             at<float>(ws, L.dwpart_sh), s);
    SimtArgs g;
    g.rows = d.tokens;
    g.A = p.x;
    g.lda = dm;
    g.B = dAs;
    g.ldb = 2 * hs;
    g.h = hs;
    g.acc_out = p.dws_gate;
    g.acc_out2 = p.dws_up;
    g.tm = tile_of(2 * hs, dm);
    g.n_mtiles = dm / g.tm;
    g.n_ntiles = 2 * hs / g.tm;
    launch_dw<DWGU, T, false>(g, (int64_t)g.n_ntiles * g.n_mtiles, d.tokens,
                              at<float>(ws, L.dwpart_sh), s);
  }
}

// the routed experts' backward
template <typename T>
void backward_routed_t(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                       cudaStream_t s) {
  const int h = d.d_hidden, dm = d.d_model, E = d.experts;
  void* dA = at<void>(ws, L.dA);
  void* gH = at<void>(ws, L.gH);
  SimtArgs z;
  z.tiles = at<int4>(ws, L.tiles);
  z.ntiles = at<int>(ws, L.ntiles);
  z.rowpair = at<int32_t>(ws, L.rowpair);
  z.top_k = d.top_k;
  z.gates = p.gates;
  z.counts = at<int>(ws, L.counts);
  z.poff = at<int>(ws, L.poff);
  SimtArgs base = z;
  z.A = p.dy;
  z.lda = dm;
  z.B = p.w_down;
  z.ldb = dm;
  z.b_estride = (int64_t)h * dm;
  z.N = h;
  z.K = dm;
  z.h = h;
  z.ag_in = p.a_gate;
  z.au_in = p.a_up;
  z.dA_out = dA;
  z.gH_out = gH;
  z.dg_part = at<float>(ws, L.dg_part);
  z.dg_ld = 2 * h / 64;  // per-pair stride of the gate-gradient partials
  z.tm = tile_of(h);     // (one partial per column tile: simt_dz_tiles(h) of them)
  z.n_ntiles = h / z.tm;
  launch<DZ, T, true>(z, z.n_ntiles * (128 / z.tm) * L.MTcap, s);

  SimtArgs x = base;
  x.A = dA;
  x.lda = 2 * h;
  x.B = p.w_gate;
  x.B2 = p.w_up;
  x.ldb = h;
  x.b_estride = (int64_t)dm * h;
  x.N = dm;
  x.K = 2 * h;
  x.h = h;
  x.slot_out = at<void>(ws, L.dxsort);
  x.ldo = dm;
  x.tm = tile_of(dm);
  x.n_ntiles = dm / x.tm;
  launch<DX, T, true>(x, x.n_ntiles * (128 / x.tm) * L.MTcap, s);

  SimtArgs w = base;
  w.A = gH;
  w.lda = h;
  w.B = p.dy;
  w.ldb = dm;
  w.acc_out = p.dw_down;
  w.ldo = dm;
  w.tm = tile_of(dm, h);
  w.n_mtiles = h / w.tm;
  w.n_ntiles = dm / w.tm;
  const int64_t krows = d.tokens * (int64_t)d.top_k / E;  // rows of an expert on average
  launch_dw<DWD, T, true>(w, (int64_t)w.n_ntiles * w.n_mtiles * E, krows,
                          at<float>(ws, L.dwpart), s);

  SimtArgs g = base;
  g.A = p.x;
  g.lda = dm;
  g.B = dA;
  g.ldb = 2 * h;
  g.h = h;
  g.acc_out = p.dw_gate;
  g.acc_out2 = p.dw_up;
  g.tm = tile_of(2 * h, dm);
  g.n_mtiles = dm / g.tm;
  g.n_ntiles = 2 * h / g.tm;
  launch_dw<DWGU, T, true>(g, (int64_t)g.n_ntiles * g.n_mtiles * E, krows,
                           at<float>(ws, L.dwpart), s);
}

}  // namespace

int simt_dz_tiles(int h) { return h / tile_of(h); }

void simt_router_logits(const moe_dims& d, const LayerPtrs& p, float* logits, cudaStream_t s) {
  if (d.dtype == MOE_BF16) router_logits_t<__nv_bfloat16>(d, p, logits, s);
  else router_logits_t<float>(d, p, logits, s);
}
void simt_grouped_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                      cudaStream_t s) {
  if (d.dtype == MOE_BF16) grouped_fwd_t<__nv_bfloat16>(d, L, mode, p, ws, s);
  else grouped_fwd_t<float>(d, L, mode, p, ws, s);
}
void simt_shared_fwd(const moe_dims& d, const Layout& L, int mode, const LayerPtrs& p, void* ws,
                     cudaStream_t s) {
  if (d.dtype == MOE_BF16) shared_fwd_t<__nv_bfloat16>(d, L, mode, p, ws, s);
  else shared_fwd_t<float>(d, L, mode, p, ws, s);
}
void simt_backward_routed(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                          cudaStream_t s) {
  if (d.dtype == MOE_BF16) backward_routed_t<__nv_bfloat16>(d, L, p, ws, s);
  else backward_routed_t<float>(d, L, p, ws, s);
}
void simt_backward_shared(const moe_dims& d, const Layout& L, const LayerPtrs& p, void* ws,
                          cudaStream_t s) {
  if (d.dtype == MOE_BF16) backward_shared_t<__nv_bfloat16>(d, L, p, ws, s);
  else backward_shared_t<float>(d, L, p, ws, s);
}

}  // namespace moe
