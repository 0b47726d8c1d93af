// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, bf16
// operands, f32 accumulators in tensor memory) for sm_103a.
//
// One persistent, warp-specialised kernel body serves every contraction of
// the forward pass and the train step (the experts_grouped_swiglu piece of
// kernel_gmm_gpu.json and the value_and_grad train step of gpu_moe_h100.json):
//
//   warp 0     producer: TMA tile loads of both operands over the expert's
//              ragged row range of the expert-sorted activations
//   warp 1     tensor-memory allocation and the MMA issuer (one thread)
//   warps 2-9  epilogue, two warps per 32-lane quarter of the accumulator
//              splitting its columns: tcgen05.ld, then the fused SwiGLU,
//              gate-weighted combine, SwiGLU backward or gradient stores.
//              bf16 tiles the epilogue reads or writes go through a
//              per-warp 32x32 staging tile in shared memory: the saved
//              pre-activations and dA, down and dX rows move with TMA loads
//              and stores; the SwiGLU outputs leave through the load/store
//              units (coalesced 16-byte copies), which keeps the TMA engine
//              for the operand loads.
//
// Tiles are 128 rows x BN columns with K blocks of 64 (one 128-byte swizzle
// row of bf16); shared memory holds a ring of STAGES operand stages and the
// accumulator is double-buffered in tensor memory so the epilogue of one
// tile overlaps the main loop of the next.  Where the tensor cores bound a
// contraction, a two-CTA cluster shares one 256-row tile (tcgen05
// cta_group::2, Cfg::PAIR): each CTA holds its 128 rows of A and half of B's
// columns, the even CTA issues the MMAs.  Every wait is bounded: a wait
// that runs out records MOE_ERR_TIMEOUT, makes the other roles leave, lets
// in-flight copies land and frees the tensor memory before returning.
#pragma once

#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tcg {

enum AKind { A_K_TMA = 0, A_MN_TMA = 2 };   // A tile K-major (rows x 64 K) or MN-major
// B tile MN-major (64 K rows x BN) or K-major; B_MN_RES: MN-major, every K
// block loaded once per CTA and kept resident (the router's W_r)
enum BKind { B_MN_TMA = 0, B_K_TMA = 1, B_MN_RES = 2 };
enum EKind { E_GU = 0, E_DOWN = 1, E_DZ = 2, E_DX = 3, E_DW = 4, E_ROUTER = 5 };

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSmemLimit = 232448;  // dynamic shared memory per block (227 KB)

// Tensor maps of one launch: the two operands (B may come from two maps,
// split along N or K) and the epilogue's bf16 outputs / inputs.
struct Maps {
  CUtensorMap a, b0, b1;
  CUtensorMap o0, o1, o2;  // DOWN / DX: output rows; DZ: dA
  CUtensorMap i0, i1;      // DZ: saved a_g, a_u
};

struct Params {
  // scheduling
  const int4* tiles = nullptr;      // routed row kinds: expert-padded tile list
  const int* ntiles_dev = nullptr;  // routed row kinds: number of tiles
  const int* counts = nullptr;      // routed DW kinds: rows per expert
  const int* poff = nullptr;        // routed DW kinds: first padded row per expert
  const int32_t* rowpair = nullptr; // padded row -> pair id (-1 = padding)
  int top_k = 1;
  int64_t rows = 0;                 // dense kinds: number of tokens
  int n_nt = 1;                     // column tiles
  int n_mt = 1;                     // DW kinds: output row tiles; dense row kinds: row tiles
  int splits = 1;                   // DW kinds: K splits
  float* part = nullptr;            // DW kinds: per-split partials [splits][E][M][ldp]
  int ldp = 0;                      //   (reduced in a fixed order by a second kernel)
                                    // routed DW kinds: per-chunk partials [chunk][M][ldp]
  int sched_units = 0;              // routed DW kinds: the work units the chunk schedule
                                    //   balances over (the whole device's, so that the
                                    //   schedule and the results do not depend on the grid)
  int* dw_tick = nullptr;           // routed DW kinds: per output tile, the chunks done;
                                    //   routed DZ zeroes them (dw_tick_n) for the DW launches
  int dw_tick_n = 0;
  int experts = 1;
  int kb_total = 0;                 // row kinds: K / 64
  int kb_split = 0;                 // dual-K B (dx): K blocks taken from the first map
  int brow_stride = 0;              // rows of a B weight matrix per expert (0: activations)
  int M = 0, N = 0;                 // DW output dims / row-kind output columns
  // epilogue
  const float* gates = nullptr;     // routed DOWN: gate per sorted row; routed DX: the router
                                    //   logit gradient of each sorted row's pair (nullable);
                                    //   router: logit offsets [E]
  const void* wrow = nullptr;       // routed DX with gates: W_r^T [E, ld_out] bf16, whose row
                                    //   e times the pair's logit gradient joins the pair's dx
  int save = 0;                     // GU: also store a_g, a_u
  void* out0 = nullptr;             // router: top-k indices [T, k]
  void* out1 = nullptr;             // router: gates [T, k]
  float* facc = nullptr;
  float* facc2 = nullptr;
  float* dg_part = nullptr;         // DZ: [pairs, dg_ld], entry 2*column-tile + half
  int dg_ld = 0;
  int ld_out = 0;
  int64_t rows_out = 0;             // GU: rows of H / a_g / a_u (load/store-unit stores)
  void* dst0 = nullptr;             // GU: H, a_g, a_u [rows_out, ld_out] bf16
  void* dst1 = nullptr;
  void* dst2 = nullptr;
  int hsplit = 0;
  int* status = nullptr;
};

// PAIR: a two-CTA cluster computes one 256 x BN tile with tcgen05's
// cta_group::2 MMA: each CTA loads its own 128 rows of A and half of B's
// columns (half the operand bytes per SM per FLOP of a single-CTA tile),
// the even CTA issues the MMAs, each CTA's epilogue drains its own rows.
template <int AK_, int BKIND_, int EK_, int BN_, bool ROUTED_, bool PAIR_ = false>
struct Cfg {
  static constexpr int AK = AK_, BKIND = BKIND_, EK = EK_, BN = BN_;
  static constexpr bool ROUTED = ROUTED_;
  static constexpr bool PAIR = PAIR_;
  static constexpr bool DW = EK == E_DW;
  static constexpr bool DUALN = EK == E_GU;
  static constexpr bool DUALK = EK == E_DX;
  static constexpr int BM = 128, BK = 64;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
  // a resident B (B_MN_RES) holds up to BRES_KB K blocks (K <= 64 * BRES_KB)
  static constexpr bool BRES = BKIND == B_MN_RES;
  static constexpr int BRES_KB = 10;
  static constexpr int STAGE_BYTES = BRES ? A_BYTES : A_BYTES + B_BYTES;
  // per-warp staging: 2 KB per bf16 32x32 tile
  // (gate/up: two tiles, a_u reuses H's slot, which leaves room for a
  // fourth operand stage)
  static constexpr int EPI_BYTES = EK == E_GU ? 2 * 2048
                                   : EK == E_DZ ? 4 * 2048
                                   : (EK == E_DOWN || EK == E_DX) ? 2048 : 0;
  // routed DW kinds keep their chunk schedule (E + 1 ints) after the barriers
  static constexpr int SCHED_BYTES = (DW && ROUTED) ? 4 * (kMaxExperts + 1) + 16 : 0;
  static constexpr int FIXED = kEpiWarps * EPI_BYTES + 1024 + 256 + SCHED_BYTES +
                               (BRES ? BRES_KB * B_BYTES : 0);
  static constexpr int STAGES = (kSmemLimit - FIXED) / STAGE_BYTES > 8
                                    ? 8
                                    : (kSmemLimit - FIXED) / STAGE_BYTES;

  static constexpr bool A_MN = AK == A_MN_TMA;
  static constexpr bool B_MN = BKIND != B_K_TMA;
  static constexpr uint32_t IDESC = tc::idesc_bf16(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + FIXED;
  static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
  static_assert(!DUALN || BN >= 128, "the gate/up tile holds 64-column halves");
  static_assert(STAGES >= 2, "shared memory");
  static_assert(!PAIR || (EK != E_ROUTER && BN >= 128), "pairs: BN >= 128, no router");
  static_assert(!BRES || (!PAIR && !DW && !DUALN), "resident B: single-CTA row kinds");
};

struct Tile {
  int e, row0, nvalid, m0, n0, kb0, kb1, nt;
  int s;   // DW kinds: K split (routed: the global chunk index)
  int ns;  // routed DW kinds: chunks of this expert (1: the tile writes the final gradient)
};

// Routed weight-gradient GEMMs reduce over each expert's rows, so a hot
// expert's tiles carry a long K range while a cold expert's are short.  The
// K range of expert e (nkb_e 64-row blocks) is cut into S_e chunks so that
// no work unit holds more than twice the average work of a CTA:
//   kb_target = max(4, 2 * ceil(sum_e nkb_e * tiles_per_expert / grid)),
//   S_e = min(kMaxChunks, ceil(nkb_e / kb_target)), at least 1.
// Uniform routing keeps S_e = 1 (no partials) unless its tiles fill less
// than half the GPU; a hot expert is cut.  choff is the prefix of S_e
// (E + 1 entries); chunk g belongs to the expert e with choff[e] <= g <
// choff[e + 1].
constexpr int kMaxChunks = 64;

// One warp: lane l takes experts l, l + 32, ... (E <= 256).
__device__ inline void dw_chunk_schedule(const int* counts, int E, int tiles_per_expert,
                                         int grid, int* choff) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = kMaxExperts / 32;
  int nkb[kPer];
  int64_t total = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    nkb[i] = e < E ? (__ldg(counts + e) + 63) / 64 : 0;
    total += nkb[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  int64_t target = 2 * ((total * tiles_per_expert + grid - 1) / grid);
  if (target < 4) target = 4;
  int base = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    int ns = (int)((nkb[i] + target - 1) / target);
    ns = e >= E ? 0 : ns < 1 ? 1 : ns > kMaxChunks ? kMaxChunks : ns;
    int incl = ns;  // inclusive scan over the 32 lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (e < E) choff[e] = base + incl - ns;
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) choff[E] = base;
}

// Tile t of the persistent schedule.  META=false skips the per-tile
// metadata loads of the routed row kinds (the MMA issuer only needs the K
// range, which is the same for every tile of those kinds).
template <class C, bool META = true>
__device__ __forceinline__ bool get_tile(const Params& p, int t, int nrow_tiles, Tile& tl,
                                         const int* choff = nullptr, int rank = 0) {
  if constexpr (!C::DW) {
    // row tiles of 128 rows; a pair takes two consecutive ones (the same
    // expert: each expert's rows are padded to 256)
    const int mu = t / p.n_nt;
    tl.nt = t % p.n_nt;
    const int mt = C::PAIR ? 2 * mu + rank : mu;
    if ((C::PAIR ? 2 * mu : mt) >= nrow_tiles) return false;
    if constexpr (C::ROUTED) {
      if constexpr (META) {
        const int4 v = tc::ld_ahead_v4(p.tiles + mt);
        tl.e = v.x;
        tl.row0 = v.y;
        tl.nvalid = v.z;
      } else {
        tl.e = tl.row0 = tl.nvalid = 0;
      }
    } else {
      tl.e = 0;
      tl.row0 = mt * C::BM;
      const int64_t left = p.rows - tl.row0;
      tl.nvalid = left < C::BM ? (left > 0 ? (int)left : 0) : C::BM;
    }
    tl.m0 = 0;
    tl.n0 = tl.nt * (C::DUALN ? C::BN / 2 : C::BN);
    tl.kb0 = 0;
    tl.kb1 = p.kb_total;
  } else {
    tl.nt = t % p.n_nt;
    int r = t / p.n_nt;
    // output row units: 128-row tiles, or 256-row tiles of a CTA pair (this
    // CTA takes the half of its rank)
    const int n_mu = C::PAIR ? p.n_mt / 2 : p.n_mt;
    const int mu = r % n_mu;
    r /= n_mu;
    const int mt = C::PAIR ? 2 * mu + rank : mu;
    int s, ns;
    int64_t ne;
    if constexpr (C::ROUTED) {
      // r is the global chunk: its expert by bisection of the schedule
      if (r >= choff[p.experts]) return false;
      int lo = 0, hi = p.experts;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (choff[mid] <= r) lo = mid;
        else hi = mid;
      }
      tl.e = lo;
      s = r - choff[lo];
      ns = choff[lo + 1] - choff[lo];
      tl.s = r;
      ne = p.counts[tl.e];
      tl.row0 = p.poff[tl.e];
    } else {
      s = r % p.splits;
      ns = p.splits;
      tl.s = s;
      tl.e = r / p.splits;
      if (tl.e >= p.experts) return false;
      ne = p.rows;
      tl.row0 = 0;
    }
    tl.ns = ns;
    const int nkb = (int)((ne + C::BK - 1) / C::BK);
    tl.kb0 = (int)((int64_t)s * nkb / ns);
    tl.kb1 = (int)((int64_t)(s + 1) * nkb / ns);
    tl.nvalid = 0;
    tl.m0 = mt * C::BM;
    tl.n0 = tl.nt * C::BN;
  }
  return true;
}

struct Shared {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t ebar[kEpiWarps];  // per epilogue warp: its staged input tiles
  uint64_t epi_bar;          // the epilogue warps' own barrier (routed DW chunk fix-up)
  uint64_t bres;             // resident B (B_MN_RES) has landed
  uint32_t tmem_base;
  volatile int abort;
  volatile int fixup;        // routed DW: this CTA finishes the tile's chunk sum
};

// CLUSTER: a barrier of a CTA pair (arrivals from the other CTA, or from
// the pair's MMA completions): polled without suspending, cluster-scope
// acquire; NAP: the many epilogue warps sleep 64 ns between polls, leaving
// the issue slots to the warps at work.
template <bool CLUSTER = false, bool NAP = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Shared* sh,
                                              int* status, int where) {
  auto try_wait = [&] {
    return CLUSTER ? tc::mbar_test_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity);
  };
  if (try_wait()) return true;
  const uint64_t t0 = tc::globaltimer();
  while (true) {
    if (CLUSTER && NAP) __nanosleep(64);
    if (try_wait()) return true;
    if (sh->abort) return false;
    if (tc::globaltimer() - t0 > 2000000000ull) {
      sh->abort = 1;
      report_error(status, MOE_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// The router's selection for one row: the top k of its E (<= EN) logits in
// the selection order (larger logit first, the lower expert index on equal
// logits) and the softmax of the selected logits.  KR > 0 (k <= KR): one
// pass, the unnormalised gates kept per thread; KR == 0: a first pass for
// the denominator and a second that repeats the selection for the gates.
template <int EN, int KR>
__device__ __forceinline__ void router_topk(const float (&lg)[64], int E, int k, int32_t* idx,
                                            float* gates) {
  auto next = [&](unsigned long long taken, float& bv) {
    int bi = -1;
    bv = 0.f;
#pragma unroll
    for (int e = 0; e < EN; ++e) {
      if (e < E && !((taken >> e) & 1ull) && (bi < 0 || better(lg[e], e, bv, bi))) {
        bv = lg[e];
        bi = e;
      }
    }
    return bi;
  };
  unsigned long long taken = 0ull;
  float top = 0.f, sum = 0.f;
  if constexpr (KR > 0) {
    // a pass loop (the unrolled selection is long: kept once in the code);
    // the unnormalised gates in a small per-thread array
    float z[KR];
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
      float bv;
      const int bi = next(taken, bv);
      taken |= 1ull << bi;
      if (r == 0) top = bv;
      z[r] = gate_exp(bv, top);
      sum += z[r];
      idx[r] = bi;
    }
#pragma unroll 1
    for (int r = 0; r < k; ++r) gates[r] = z[r] / sum;
  } else {
    for (int r = 0; r < k; ++r) {
      float bv;
      const int bi = next(taken, bv);
      taken |= 1ull << bi;
      if (r == 0) top = bv;
      sum += gate_exp(bv, top);
      idx[r] = bi;
    }
    taken = 0ull;
    for (int r = 0; r < k; ++r) {
      float bv;
      taken |= 1ull << next(taken, bv);
      gates[r] = gate_exp(bv, top) / sum;
    }
  }
}

// The epilogue warps' own barrier: one arrival per warp, a bounded wait.
__device__ __forceinline__ bool epi_sync(Shared* sh, uint32_t& phase, int* status) {
  if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&sh->epi_bar);
  const bool ok = wait_or_abort(&sh->epi_bar, phase, sh, status, 600);
  phase ^= 1;
  return ok;
}

// Routed DW tile of an expert cut into ns > 1 K chunks: after storing its
// partial, the CTA takes a ticket; the one that finishes the tile's last
// chunk (any order) sums the ns partials in chunk order into the gradient
// and resets the ticket.  Returns false when a wait ran out.
template <class C>
__device__ bool dw_chunk_fixup(const Params& p, const Tile& tl, const int* choff, Shared* sh,
                               int row, int half, uint32_t& phase) {
  __threadfence();  // this thread's partial stores before the ticket
  if (!epi_sync(sh, phase, p.status)) return false;
  if (threadIdx.x == 64) {
    const int slot = (tl.e * p.n_mt + tl.m0 / C::BM) * p.n_nt + tl.nt;
    const int done = atomicAdd(p.dw_tick + slot, 1) + 1;
    const bool last = done == tl.ns;
    if (last) p.dw_tick[slot] = 0;  // ready for the next launch
    __threadfence();
    sh->fixup = last ? 1 : 0;
  }
  if (!epi_sync(sh, phase, p.status)) return false;
  if (!sh->fixup) return true;
  const int om = tl.m0 + row;
  if (om >= p.M) return true;
  float* base = p.facc;
  int ncol = tl.n0, ld = p.N;
  if (p.hsplit > 0) {
    ld = p.hsplit;
    if (tl.n0 >= p.hsplit) {
      base = p.facc2;
      ncol = tl.n0 - p.hsplit;
    }
  }
  float* dst = base + ((int64_t)tl.e * p.M + om) * ld + ncol;
  const int g0 = choff[tl.e];
  const int64_t cstride = (int64_t)p.M * p.ldp;
  const float* src = p.part + ((int64_t)g0 * p.M + om) * p.ldp + tl.n0;
#pragma unroll 1
  for (int c = half; c < C::BN / 32; c += 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < tl.ns; ++s) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + s * cstride + 32 * c + 4 * i));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      *reinterpret_cast<float4*>(dst + 32 * c + 4 * i) = acc;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// A staged 32x32 bf16 tile (64-byte swizzle) to rows y0.. / columns x.. of a
// row-major [rows, ld] bf16 array: lane l copies 16 bytes of rows l/4,
// l/4 + 8, ... (four lanes per 64-byte row piece), rows past `rows` skipped.
__device__ __forceinline__ void staged_copy_out(const uint8_t* tile, void* dst, int y0, int x,
                                                int ld, int64_t rows, int lane) {
  const int q = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i;
    const uint4 v = *reinterpret_cast<const uint4*>(tile + tc::sw64_off(r, q));
    if ((int64_t)y0 + r < rows)
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dst) +
                                ((int64_t)y0 + r) * ld + x + 8 * q) = v;
  }
}

// One thread's row of a 64-byte-swizzled 32x32 staging tile as 16 bf16 pairs.
__device__ __forceinline__ void stage_read_packed(const uint8_t* tile, int r, uint32_t (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + tc::sw64_off(r, k));
    w[4 * k] = u.x;
    w[4 * k + 1] = u.y;
    w[4 * k + 2] = u.z;
    w[4 * k + 3] = u.w;
  }
}

// One thread's row of 32 bf16 already packed in pairs (bf16x2_rn).
__device__ __forceinline__ void stage_write_packed(uint8_t* tile, int r, const uint32_t (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(tile + tc::sw64_off(r, k)) =
        make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

__device__ __forceinline__ void stage_write_row(uint8_t* tile, int r, const float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(tile + tc::sw64_off(r, k)) =
        make_uint4(pack_bf16(v[8 * k], v[8 * k + 1]), pack_bf16(v[8 * k + 2], v[8 * k + 3]),
                   pack_bf16(v[8 * k + 4], v[8 * k + 5]), pack_bf16(v[8 * k + 6], v[8 * k + 7]));
}

template <class C>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ Maps m, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sBres = smem + C::STAGES * C::STAGE_BYTES;  // resident B (B_MN_RES)
  uint8_t* epi = sBres + (C::BRES ? C::BRES_KB * C::B_BYTES : 0);
  Shared* sh = reinterpret_cast<Shared*>(epi + kEpiWarps * C::EPI_BYTES);
  int* choff = reinterpret_cast<int*>(sh + 1);  // routed DW kinds: the chunk schedule
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work units: one per CTA, or one per CTA pair (both CTAs walk the same units)
  const int rank = C::PAIR ? (int)tc::cluster_ctarank() : 0;
  const int u0 = C::PAIR ? (int)tc::cluster_id_x() : (int)blockIdx.x;
  const int us = C::PAIR ? (int)tc::ncluster_x() : (int)gridDim.x;

  if (threadIdx.x == 0) {
    // a pair's even CTA: its full barriers count both CTAs' operand bytes
    // (one arrival, its own producer's), its accumulator-empty barriers both
    // CTAs' epilogue warps
    const int both = C::PAIR && rank == 0 ? 2 : 1;
    for (int s = 0; s < C::STAGES; ++s) {
      tc::mbar_init(&sh->full[s], 1);
      tc::mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sh->tfull[a], 1);
      tc::mbar_init(&sh->tempty[a], kEpiWarps * both);
    }
    for (int w = 0; w < kEpiWarps; ++w) tc::mbar_init(&sh->ebar[w], 1);
    tc::mbar_init(&sh->epi_bar, kEpiWarps);
    tc::mbar_init(&sh->bres, 1);
    sh->abort = 0;
    tc::fence_barrier_init();
  }
  if constexpr (C::DW && C::ROUTED) {
    if (warp == 2)  // an epilogue warp (idle until the first tile is ready)
      dw_chunk_schedule(p.counts, p.experts, (C::PAIR ? p.n_mt / 2 : p.n_mt) * p.n_nt,
                        p.sched_units > 0 ? p.sched_units : us, choff);
  }
  if constexpr (C::EK == E_DZ && C::ROUTED) {
    // the chunk tickets of the weight-gradient launches that follow start at 0
    if (blockIdx.x == 0 && p.dw_tick)
      for (int i = threadIdx.x; i < p.dw_tick_n; i += blockDim.x) p.dw_tick[i] = 0;
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&m.a);
    tc::tma_prefetch_desc(&m.b0);
    tc::tma_prefetch_desc(&m.b1);
  }
  if constexpr (C::PAIR) {
    // both CTAs' barriers are initialised before either signals the other's
    tc::cluster_sync();
    if (warp == 1) {
      tc::tmem_alloc_pair(&sh->tmem_base, C::TMEM_COLS);
      tc::tmem_relinquish_pair();
    }
  } else if (warp == 1) {
    tc::tmem_alloc(&sh->tmem_base, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  int nrow_tiles = p.n_mt;
  if constexpr (C::ROUTED && !C::DW) nrow_tiles = p.ntiles_dev[0];

  bool aborted = false;
  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      if constexpr (C::BRES) {  // every K block of B once, before the first tile
        tc::mbar_arrive_expect_tx(&sh->bres, p.kb_total * C::B_BYTES);
        for (int kb = 0; kb < p.kb_total; ++kb)
          tc::tma_load_2d(sBres + kb * C::B_BYTES, &m.b0, &sh->bres, 0, kb * C::BK);
      }
      int stage = 0;
      uint32_t phase = 0;
      // the next tile's metadata is read while this tile's loads are issued
      Tile tl, tn;
      int t = u0;
      bool have = get_tile<C>(p, t, nrow_tiles, tl, choff, rank);
      for (; !aborted && have; t += us, tl = tn) {
        have = get_tile<C>(p, t + us, nrow_tiles, tn, choff, rank);
        int brow0 = 0;
        if constexpr (C::ROUTED && !C::DW) brow0 = tl.e * p.brow_stride;
        if constexpr (C::DW) brow0 = tl.row0;
        for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
          if (!wait_or_abort<C::PAIR>(&sh->empty[stage], phase ^ 1, sh, p.status, 100)) {
            aborted = true;
            break;
          }
          uint8_t* sA = smem + stage * C::STAGE_BYTES;
          uint8_t* sB = sA + C::A_BYTES;
          uint64_t* fb = &sh->full[stage];
          // a pair: both CTAs' copies complete on the even CTA's barrier,
          // which expects the bytes of both
          const uint32_t fbc = C::PAIR ? tc::peer_addr(fb, 0) : 0u;
          if (!C::PAIR) tc::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          else if (rank == 0) tc::mbar_arrive_expect_tx(fb, 2 * C::STAGE_BYTES);
          auto load = [&](void* dst, const CUtensorMap* mp, int x, int y) {
            if constexpr (C::PAIR) tc::tma_load_2d_pair(dst, mp, fbc, x, y);
            else tc::tma_load_2d(dst, mp, fb, x, y);
          };
          // ---- A ----
          if constexpr (C::AK == A_K_TMA) {
            load(sA, &m.a, kb * C::BK, tl.row0);
          } else {  // MN-major: two 64-column blocks of 64 K rows
            const int krow = (C::DW ? tl.row0 : 0) + kb * C::BK;
            load(sA, &m.a, tl.m0, krow);
            load(sA + 8192, &m.a, tl.m0 + 64, krow);
          }
          // ---- B ----  (a pair holds half of B's columns per CTA; gate/up:
          // the even CTA the gate half, the odd CTA the up half)
          constexpr int BNL = C::PAIR ? C::BN / 2 : C::BN;
          const int nb0 = tl.n0 + (C::PAIR && !C::DUALN ? rank * BNL : 0);
          if constexpr (C::BRES) {
          } else if constexpr (C::BKIND == B_MN_TMA) {
#pragma unroll
            for (int j = 0; j < BNL / 64; ++j) {
              const CUtensorMap* mp = &m.b0;
              int x = nb0 + 64 * j;
              if constexpr (C::DUALN && C::PAIR) {
                if (rank) mp = &m.b1;
              } else if constexpr (C::DUALN) {
                const bool second = j >= C::BN / 128;
                x = tl.n0 + 64 * (second ? j - C::BN / 128 : j);
                if (second) mp = &m.b1;
              }
              load(sB + j * 8192, mp, x, brow0 + kb * C::BK);
            }
          } else {  // K-major: BNL rows of 64 K (the tensor map's box)
            const bool second = C::DUALK && kb >= p.kb_split;
            const int x = (second ? kb - p.kb_split : kb) * C::BK;
            load(sB, second ? &m.b1 : &m.b0, x, brow0 + nb0);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && C::PAIR && rank == 1) {
    // odd CTA of a pair: the even CTA issues the pair's MMAs
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    int stage = 0, acc = 0;
    uint32_t phase = 0, aphase = 0;
    if constexpr (C::BRES) {
      if (!wait_or_abort(&sh->bres, 0, sh, p.status, 310)) aborted = true;
    }
    Tile tl;
    for (int t = u0; !aborted && get_tile<C, false>(p, t, nrow_tiles, tl, choff, rank);
         t += us) {
      if (!wait_or_abort<C::PAIR>(&sh->tempty[acc], aphase ^ 1, sh, p.status, 200)) {
        aborted = true;
        break;
      }
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::BN;
      for (int kb = tl.kb0; kb < tl.kb1; ++kb) {
        if (!wait_or_abort<C::PAIR>(&sh->full[stage], phase, sh, p.status, 300)) {
          aborted = true;
          break;
        }
        tc::tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = tc::smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t b0 = C::BRES ? tc::smem_u32(sBres + kb * C::B_BYTES) : a0 + C::A_BYTES;
#pragma unroll
          for (int s = 0; s < C::BK / 16; ++s) {
            const uint64_t ad = C::A_MN ? tc::sw128_desc(a0 + s * 2048, 8192, 1024)
                                        : tc::sw128_desc(a0 + s * 32, 0, 1024);
            const uint64_t bd = C::B_MN ? tc::sw128_desc(b0 + s * 2048, 8192, 1024)
                                        : tc::sw128_desc(b0 + s * 32, 0, 1024);
            const uint32_t accum = (kb > tl.kb0 || s > 0) ? 1u : 0u;
            if constexpr (C::PAIR) tc::mma_bf16_pair(d_tmem, ad, bd, C::IDESC, accum);
            else tc::mma_bf16(d_tmem, ad, bd, C::IDESC, accum);
          }
          if constexpr (C::PAIR) tc::mma_commit_pair(&sh->empty[stage]);
          else tc::mma_commit(&sh->empty[stage]);
        }
        __syncwarp();
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (aborted) break;
      if (lane == 0) {
        if constexpr (C::PAIR) tc::mma_commit_pair(&sh->tfull[acc]);
        else tc::mma_commit(&sh->tfull[acc]);
      }
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1;
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    // warp w >= 2: lane quarter q = w % 4 (the tcgen05.ld lane window of the
    // warp), column half = (w - 2) / 4: the two warps of a quarter take
    // alternate 32-column chunks
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    const int row = 32 * q + lane;
    uint8_t* stg = epi + ew * C::EPI_BYTES;  // this warp's staging tiles
    uint64_t* ebar = &sh->ebar[ew];
    uint32_t ephase = 0;
    int acc = 0;
    uint32_t aphase = 0, epi_phase = 0;
    Tile tl, tn;
    int t = u0;
    bool have = get_tile<C>(p, t, nrow_tiles, tl, choff, rank);
    // DZ: saved a_g / a_u of this warp's first chunk, loaded ahead of the MMA
    if constexpr (C::EK == E_DZ) {
      if (have && lane == 0) {
        tc::mbar_arrive_expect_tx(ebar, 4096);
        tc::tma_load_2d(stg, &m.i0, ebar, tl.n0 + 32 * half, tl.row0 + 32 * q);
        tc::tma_load_2d(stg + 2048, &m.i1, ebar, tl.n0 + 32 * half, tl.row0 + 32 * q);
      }
    }
    // routed DOWN: the gate of this thread's row; routed DX: its pair's
    // router logit gradient; read a tile ahead (after the previous tile's
    // first chunk)
    constexpr bool ROWSC = C::ROUTED && (C::EK == E_DOWN || C::EK == E_DX);
    const bool rowsc = ROWSC && p.gates;
    float gt_next = 0.f;
    if constexpr (ROWSC) {
      if (rowsc && have && row < tl.nvalid) gt_next = p.gates[(int64_t)tl.row0 + row];
    }
    // routed DX with the router term: the entries of W_r^T[e] under this
    // warp's chunks of a tile (c = half, half + 2, ...), spread over the
    // lanes (lane l: 8 entries at 8 (l % 4) of its (l / 4)-th chunk) and
    // read a tile ahead; each chunk takes its 32 entries by shuffles
    constexpr int NCH = C::BN / 64 > 0 ? C::BN / 64 : 1;  // chunks per warp and tile
    int4 wr_cur = make_int4(0, 0, 0, 0), wr_next = make_int4(0, 0, 0, 0);
    auto load_wr = [&](const Tile& x) {
      if (lane < 4 * NCH) {
        const int c = half + 2 * (lane >> 2);
        wr_next = tc::ld_ahead_v4(
            reinterpret_cast<const int4*>(reinterpret_cast<const __nv_bfloat16*>(p.wrow) +
                                          (int64_t)x.e * p.ld_out + x.n0 + 32 * c) +
            (lane & 3));
      }
    };
    if constexpr (C::ROUTED && C::EK == E_DX) {
      if (rowsc && have) load_wr(tl);
    }
    while (have && !aborted) {
      // the next tile's metadata is read while this one is processed
      const bool have_next = get_tile<C>(p, t + us, nrow_tiles, tn, choff, rank);
      // per-row metadata of this tile (routed kinds): issued before the wait
      int32_t pr = -1;
      float gt = 1.f;
      if constexpr (C::ROUTED && C::EK == E_DZ) {
        if (row < tl.nvalid) pr = p.rowpair[(int64_t)tl.row0 + row];
      }
      if constexpr (ROWSC) gt = gt_next;
      if constexpr (C::ROUTED && C::EK == E_DX) wr_cur = wr_next;
      if (!wait_or_abort<C::PAIR, true>(&sh->tfull[acc], aphase, sh, p.status, 400)) {
        aborted = true;
        break;
      }
      tc::tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(32 * q) << 16) + acc * C::BN;
      const bool has_k = tl.kb1 > tl.kb0;
      const int yrow = tl.row0 + 32 * q;  // first row of this warp's tiles
      // dense row kinds: a pair's odd CTA may hold a tile past the last token
      // (odd tile count); its stores are skipped
      const bool ystore = C::ROUTED || (int64_t)yrow < p.rows;

      if constexpr (C::EK == E_GU) {
        // H = silu(a_g) * a_u with a_g, a_u rounded to bf16 first (the values
        // a backward pass reads back), in float pairs; staged 32x32 tiles
        // copied out by the load/store units
#pragma unroll 1
        for (int c = half; c < C::BN / 64; c += 2) {
          uint32_t g[32], u[32];
          tc::tmem_ld32(tacc + 32 * c, g);
          tc::tmem_ld32(tacc + C::BN / 2 + 32 * c, u);
          tc::tmem_ld_wait();
          uint32_t gp[16], up[16], hp[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            gp[j] = tc::bf16x2_rn(__uint_as_float(g[2 * j]), __uint_as_float(g[2 * j + 1]));
            up[j] = tc::bf16x2_rn(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1]));
            const uint64_t gx = tc::bf16x2_to_f2(gp[j]);
            float h0, h1;
            tc::f2_split(tc::f2_mul(tc::f2_mul(gx, tc::f2_sigmoid(gx)), tc::bf16x2_to_f2(up[j])),
                         h0, h1);
            hp[j] = tc::bf16x2_rn(h0, h1);
          }
          __syncwarp();  // the previous chunk's copies have read the staging
          stage_write_packed(stg, lane, hp);
          if (p.save) stage_write_packed(stg + 2048, lane, gp);
          __syncwarp();
          const int x = tl.n0 + 32 * c;
          staged_copy_out(stg, p.dst0, yrow, x, p.ld_out, p.rows_out, lane);
          if (p.save) {
            staged_copy_out(stg + 2048, p.dst1, yrow, x, p.ld_out, p.rows_out, lane);
            __syncwarp();  // H's copies have read the first slot
            stage_write_packed(stg, lane, up);
            __syncwarp();
            staged_copy_out(stg, p.dst2, yrow, x, p.ld_out, p.rows_out, lane);
          }
        }
      } else if constexpr (C::EK == E_DOWN || C::EK == E_DX) {
        // one output row per sorted row, stored by TMA as bf16 tiles:
        //   DOWN: gate * (H W_down), the pair's share of its token's output
        //         (the shared expert: its whole output row)
        //   DX:   [dA_g | dA_u] [W_gate | W_up]^T, the pair's share of dx,
        //         plus (routed, with the router term) dl_pair W_r[:, e]^T
        // the combine gathers the k shares of a token in a fixed order
        const float sc = C::EK == E_DOWN ? gt : 1.f;
#pragma unroll 1
        for (int c = half; c < C::BN / 32; c += 2) {
          int4 w4[4];  // the chunk's 32 entries of W_r^T[e] (the same for every row)
          if constexpr (C::ROUTED && C::EK == E_DX) {
            if (rowsc) {
              const int src = 4 * ((c - half) >> 1);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                w4[k4].x = __shfl_sync(0xffffffffu, wr_cur.x, src + k4);
                w4[k4].y = __shfl_sync(0xffffffffu, wr_cur.y, src + k4);
                w4[k4].z = __shfl_sync(0xffffffffu, wr_cur.z, src + k4);
                w4[k4].w = __shfl_sync(0xffffffffu, wr_cur.w, src + k4);
              }
              if (c == half && have_next) load_wr(tn);
            }
          }
          uint32_t v[32];
          tc::tmem_ld32(tacc + 32 * c, v);
          tc::tmem_ld_wait();
          float o[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = sc * __uint_as_float(v[i]);
          if constexpr (C::ROUTED && C::EK == E_DX) {
            if (rowsc) {
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const uint32_t wv[4] = {(uint32_t)w4[k4].x, (uint32_t)w4[k4].y,
                                        (uint32_t)w4[k4].z, (uint32_t)w4[k4].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  o[8 * k4 + 2 * j] = fmaf(gt, __uint_as_float(wv[j] << 16), o[8 * k4 + 2 * j]);
                  o[8 * k4 + 2 * j + 1] =
                      fmaf(gt, __uint_as_float(wv[j] & 0xFFFF0000u), o[8 * k4 + 2 * j + 1]);
                }
              }
            }
          }
          if (lane == 0) tc::bulk_wait_read0();
          __syncwarp();
          stage_write_row(stg, lane, o);
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && ystore) {
            tc::tma_store_2d(&m.o0, stg, tl.n0 + 32 * c, yrow);
            tc::bulk_commit();
          }
          if constexpr (ROWSC) {
            if (rowsc && c == half)
              gt_next = have_next && row < tn.nvalid
                            ? tc::ld_ahead_f32(p.gates + (int64_t)tn.row0 + row)
                            : 0.f;
          }
        }
      } else if constexpr (C::EK == E_DZ) {
        // the routed rows of dy arrive scaled by their pair's gate, so the
        // accumulator holds dH = g (dy W_down^T) (the shared expert: g = 1);
        // SwiGLU backward from the saved pre-activations (TMA-staged); the
        // partial <dH, H> = g dg over these columns; dA tiles stored by TMA
        const int h = p.ld_out;
        uint64_t dgp2 = tc::f2(0.f, 0.f);  // <dH, H> over even / odd columns
#pragma unroll 1
        for (int c = half; c < C::BN / 32; c += 2) {
          uint32_t zv[32];
          tc::tmem_ld32(tacc + 32 * c, zv);
          tc::tmem_ld_wait();
          if (!wait_or_abort(ebar, ephase, sh, p.status, 500)) {
            aborted = true;
            break;
          }
          ephase ^= 1;
          uint32_t wg[16], wu[16];
          stage_read_packed(stg, lane, wg);
          stage_read_packed(stg + 2048, lane, wu);
          // the copies below overwrite these staging tiles: every lane's reads
          // must have returned first, so an instruction that needs all of
          // them (a branch that is never taken) stands before the barrier
          {
            uint32_t landed = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) landed ^= wg[j] ^ wu[j];
            if (landed == 0x9e3779b9u && p.top_k < 0) sh->abort = sh->abort;
          }
          __syncwarp();
          // the next input tiles of this warp: next chunk, or the first chunk
          // of the next tile
          if (lane == 0) {
            const bool more = c + 2 < C::BN / 32;
            if (more || have_next) {
              const int nx = more ? tl.n0 + 32 * (c + 2) : tn.n0 + 32 * half;
              const int ny = more ? yrow : tn.row0 + 32 * q;
              tc::mbar_arrive_expect_tx(ebar, 4096);
              tc::tma_load_2d(stg, &m.i0, ebar, nx, ny);
              tc::tma_load_2d(stg + 2048, &m.i1, ebar, nx, ny);
            }
          }
          // in float pairs: s = sigmoid(a_g), H = bf16(a_g s a_u) as the
          // forward stored it, dA_u = dH a_g s, dA_g = dH a_u s (1 + a_g (1 - s))
          uint32_t dagp[16], daup[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint64_t ag = tc::bf16x2_to_f2(wg[j]), au = tc::bf16x2_to_f2(wu[j]);
            const uint64_t dh = tc::f2(__uint_as_float(zv[2 * j]), __uint_as_float(zv[2 * j + 1]));
            const uint64_t sg = tc::f2_sigmoid(ag);
            const uint64_t sl = tc::f2_mul(ag, sg);
            float h0, h1;
            tc::f2_split(tc::f2_mul(sl, au), h0, h1);
            dgp2 = tc::f2_fma(dh, tc::bf16x2_to_f2(tc::bf16x2_rn(h0, h1)), dgp2);
            float a0, a1;
            tc::f2_split(tc::f2_mul(dh, sl), a0, a1);
            daup[j] = tc::bf16x2_rn(a0, a1);
            const uint64_t oms = tc::f2_fma(sg, tc::f2(-1.f, -1.f), tc::f2(1.f, 1.f));
            const uint64_t inner = tc::f2_fma(ag, oms, tc::f2(1.f, 1.f));
            tc::f2_split(tc::f2_mul(tc::f2_mul(tc::f2_mul(dh, au), sg), inner), a0, a1);
            dagp[j] = tc::bf16x2_rn(a0, a1);
          }
          if (lane == 0) tc::bulk_wait_read0();
          __syncwarp();
          stage_write_packed(stg + 4096, lane, dagp);
          stage_write_packed(stg + 6144, lane, daup);
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && ystore) {
            const int x = tl.n0 + 32 * c;
            tc::tma_store_2d(&m.o0, stg + 4096, x, yrow);
            tc::tma_store_2d(&m.o0, stg + 6144, h + x, yrow);
            tc::bulk_commit();
          }
        }
        if (aborted) break;
        if (C::ROUTED && pr >= 0) {
          float d0, d1;
          tc::f2_split(dgp2, d0, d1);
          p.dg_part[(int64_t)pr * p.dg_ld + 2 * tl.nt + half] = d0 + d1;
        }
      } else if constexpr (C::EK == E_ROUTER) {
        // router: one token per thread of the first four epilogue warps; its
        // E logits come straight from tensor memory, the top-k selection and
        // the softmax of the selected logits run in registers
        if (half == 0) {
          float lg[C::BN];
#pragma unroll
          for (int c = 0; c < C::BN / 32; ++c) {
            uint32_t v[32];
            tc::tmem_ld32(tacc + 32 * c, v);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) lg[32 * c + i] = __uint_as_float(v[i]);
          }
          const int E = p.N, k = p.top_k;
          if (p.gates) {  // the router bias (a fixed offset per expert)
#pragma unroll
            for (int e = 0; e < C::BN; ++e)
              if (e < E) lg[e] += __ldg(p.gates + e);
          }
          if (row < tl.nvalid) {
            const int64_t t = (int64_t)tl.row0 + row;
            if (p.facc) {
              float4* lo = reinterpret_cast<float4*>(p.facc + t * E);
#pragma unroll
              for (int e4 = 0; e4 < C::BN / 4; ++e4)
                if (4 * e4 < E) lo[e4] = make_float4(lg[4 * e4], lg[4 * e4 + 1], lg[4 * e4 + 2], lg[4 * e4 + 3]);
            }
            int32_t* idx = reinterpret_cast<int32_t*>(p.out0) + t * k;
            float* gates = reinterpret_cast<float*>(p.out1) + t * k;
            if (k <= 8 && E <= 8) router_topk<8, 8>(lg, E, k, idx, gates);
            else if (k <= 8 && E <= 16) router_topk<16, 8>(lg, E, k, idx, gates);
            else if (k <= 8 && E <= 32) router_topk<32, 8>(lg, E, k, idx, gates);
            else if (k <= 8) router_topk<64, 8>(lg, E, k, idx, gates);
            else router_topk<64, 0>(lg, E, k, idx, gates);
          }
        }
      } else {  // E_DW: one expert's gradient tile (rows m0.., columns n0..)
        const int om = tl.m0 + row;
        float* base = p.facc;
        int ncol = tl.n0, ld = p.N;
        if (p.hsplit > 0) {
          ld = p.hsplit;
          if (tl.n0 >= p.hsplit) {
            base = p.facc2;
            ncol = tl.n0 - p.hsplit;
          }
        }
        // one split's partial (reduced later in split order) or the final
        // gradient; every element of the tile is written once (zeros when
        // this split's K range is empty)
        float* dst;
        if constexpr (C::ROUTED) {  // a chunk's partial, or the final gradient for one chunk
          dst = tl.ns > 1 ? p.part + ((int64_t)tl.s * p.M + om) * p.ldp + tl.n0
                          : base + ((int64_t)tl.e * p.M + om) * ld + ncol;
        } else {
          dst = p.part ? p.part + ((int64_t)tl.s * p.experts * p.M + (int64_t)tl.e * p.M + om) *
                                      p.ldp + tl.n0
                       : base + ((int64_t)tl.e * p.M + om) * ld + ncol;
        }
#pragma unroll 1
        for (int c = half; c < C::BN / 32; c += 2) {
          uint32_t v[32];
          if (has_k) {
            tc::tmem_ld32(tacc + 32 * c, v);
            tc::tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          if (om < p.M) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 f = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                           __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
              *reinterpret_cast<float4*>(dst + 32 * c + 4 * i) = f;
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        // a pair's MMA issuer (even CTA) waits for both CTAs' epilogues
        if (C::PAIR && rank == 1) tc::mbar_arrive_cluster(tc::peer_addr(&sh->tempty[acc], 0));
        else tc::mbar_arrive(&sh->tempty[acc]);
      }
      if constexpr (C::DW && C::ROUTED) {
        if (tl.ns > 1 && !dw_chunk_fixup<C>(p, tl, choff, sh, row, half, epi_phase)) {
          aborted = true;
          break;
        }
      }
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1;
      }
      t += us;
      tl = tn;
      have = have_next;
    }
    if constexpr (C::EPI_BYTES > 0) {
      if (lane == 0) tc::bulk_wait0();  // this warp's tile stores are complete
      __syncwarp();
    }
  }

  if (aborted || sh->abort) {
    // let copies and MMAs already in flight land before the memory goes away
    const uint64_t t0 = tc::globaltimer();
    while (tc::globaltimer() - t0 < 2000000ull) {
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if constexpr (C::PAIR) {
    // neither CTA leaves while the even CTA's MMAs may still touch the odd
    // CTA's shared or tensor memory, or the odd CTA may still arrive on the
    // even CTA's barriers
    tc::cluster_sync();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  } else {
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();
int sm_count();    // SMs of the current device
int launch_sms();  // SMs the calling thread's launches may fill (moe_set_sm_limit)

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, out-of-bounds
// elements read as zero (stores outside are dropped).  Operand tiles use the
// 128-byte swizzle (box_cols = 64); the epilogue's 32x32 staging tiles use
// the 64-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows);
bool make_map_sw64(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols);

template <class C>
void launch_tc(const Maps& maps, const Params& p, int64_t max_tiles, const char* name,
               cudaStream_t s) {
  if (max_tiles <= 0) return;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(tc_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         C::SMEM_BYTES);
    attr = true;
  }
  const int sms = launch_sms();
  if constexpr (C::PAIR) {
    // max_tiles counts pair units; two CTAs (one cluster) per unit, no more
    // clusters than can be resident at once (an SM whose partner SM is not
    // available takes no pair, and a cluster left for a second wave would
    // double the persistent schedule's time)
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeClusterDimension;
    attr1[0].val.clusterDim.x = 2;
    attr1[0].val.clusterDim.y = 1;
    attr1[0].val.clusterDim.z = 1;
    cfg.attrs = attr1;
    cfg.numAttrs = 1;
    static int resident = 0;
    if (resident == 0) {
      cfg.gridDim = dim3(sm_count(), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<C>, &cfg) != cudaSuccess || n < 1)
        n = sm_count() / 2;
      resident = n;
    }
    int cap = resident < sms / 2 ? resident : sms / 2;
    if (cap < 1) cap = 1;
    const int pairs = (int)(max_tiles < cap ? max_tiles : cap);
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    MOE_LAUNCH(name, s, cudaLaunchKernelEx(&cfg, tc_gemm_kernel<C>, maps, p));
  } else {
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    MOE_LAUNCH(name, s, tc_gemm_kernel<C><<<grid, kThreads, C::SMEM_BYTES, s>>>(maps, p));
  }
}

}  // namespace tcg
}  // namespace moe
