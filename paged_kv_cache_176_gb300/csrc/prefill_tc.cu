// prefill_tc.cu -- chunked-prefill attention on the tcgen05 tensor cores (bf16).
//
// A prefill chunk of q_len tokens of sequence s (context ctx, which includes
// the chunk) attends causally over absolute positions: query row i sits at
// position ctx - q_len + i and sees keys 0 .. that position, i.e. the cached
// keys of all earlier chunks plus its own tokens up to itself ("Chunked
// Prefill" glossary page, how chunked prefill works: the mask
// ones(end - start, end).tril(diagonal = start)). Keys and values are gathered
// through the sequence's block table (K_r = gather(K_pool, table_r), the
// gather figure of the "C13 L2 serving" page).
//
// GB300 design: one CTA per unit of one KV head, a unit being one or two Q
// tiles of 128 rows (128/G consecutive tokens x the G query heads that share
// the KV head), so that one K/V tile in shared memory serves up to 256 rows.
//  * Warp 0 moves the Q tiles once and then K tiles of 128 keys (8 pool
//    blocks) into a two-stage ring, warp 10 moves V tiles into a two-stage
//    ring; each block is one 3-D tiled TMA copy (64 head-dim columns x 16
//    tokens, 128-byte swizzle) straight out of the paged pool, so the gather
//    costs no extra pass.
//  * Warp 1 owns all 512 TMEM columns (S and O of each Q tile, 128 columns
//    each) and issues the MMAs from one thread: S_x = Q_x K^T (128 x 128,
//    fp32) and O_x += P_x V with P_x read from TMEM (the A operand of a
//    TS-MMA) and V (128 keys x head_dim) from shared memory. The two Q tiles
//    alternate: while the softmax of one tile runs, the tensor pipe works on
//    the other's products, and S_x(j+1) follows P_x(j) V(j) in the pipe.
//  * Warps 2-5 (Q tile 0) and 6-9 (Q tile 1) hold one thread per query row.
//    Each reads its row of S from TMEM, 64 keys at a time, and writes
//    P = 2^(s - m) of those keys as bf16 pairs over scores it has read, m
//    being its running max in the log2 domain. The max moves only when a
//    score exceeds it by more than 8 (lazy rescaling), and a sum bounds every
//    weight in it: while a half's sum stays at or below 2^8 no score of it
//    passed m + 8, so the tile needs no max pass. Only otherwise (and on the
//    first tile) is the max of the scores still in TMEM taken and the half
//    redone with it (P of the first half, already stored, rescaled in place),
//    O rescaled in TMEM when the max moved. Masked keys get weight 0.
//  * On the last key tile the rows of Q tile 0 zero the value rows that lie
//    past the context or past the loaded blocks, before P_0 goes to the MMA,
//    so stale or NaN slots never reach the result.
//  * Units run longest first: every CTA finds the unit of its rank in the
//    order of decreasing key-tile count from the chunk lengths alone.
//  * Every wait is bounded; a timeout sets PA_STATUS_TIMEOUT, the roles stop,
//    wait (bounded) for their copies and MMAs in flight, and the CTA releases
//    its TMEM and leaves.
#include <cuda.h>
#include <algorithm>
#include <cuda_runtime.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace pa {
namespace {

constexpr int kD = 128;              // head_dim of the tensor-core path
constexpr int kRowsTile = 128;       // query rows per Q tile (MMA M)
constexpr int kKeysTile = 128;       // keys per tile (MMA N of Q K^T)
constexpr int kBlocksTile = kKeysTile / kBlockSize;
constexpr int kThreadsTc = 352;      // warp 0 Q/K loads, warp 1 MMA, warps 2-9 softmax, warp 10 V loads
constexpr int kVWarp = 10;
constexpr int kHalf = 16384;         // one 64-column half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalf;
constexpr int kKStages = 2;          // K is released as soon as both S = Q K^T are done
constexpr int kVStages = 2;          // V is released after both O += P V

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                               // Q tiles 0 and 1
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBar = kOffV + kVStages * kTileBytes;
constexpr int kSmemTc = kOffBar + 256 + 1024;          // + barriers + alignment slack
constexpr int kMaxPrefixSeqs = 8191;                   // sequences (groups) per launch

// TMEM columns: S of Q tile x at 128 x, O of Q tile x at 256 + 128 x
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int x) { return static_cast<uint32_t>(x) * 128u; }
__device__ __forceinline__ uint32_t col_o(int x) { return 256u + static_cast<uint32_t>(x) * 128u; }

struct TcParams {
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  const int32_t* block_tables;
  void* out;
  int num_seqs, num_rows, hq, hkv, group, max_blocks;
  int q_tiles;  // Q tiles per unit: 1 or 2
  int64_t num_blocks;
  float scale_log2;
  int* d_status;
  int prefix_mode;  // cascade decode: groups of decode rows over a shared prefix
  float2* pre_ml;
  float* pre_acc;
};

struct TcBarriers {
  uint64_t q_full;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];   // [Q tile]: S = Q K^T of the current key tile is in TMEM
  uint64_t p_full[2];   // [Q tile]: its P is in TMEM (one arrival per softmax warp)
  uint64_t pv_done[2];  // [Q tile]: O += P V of the current key tile is complete
  uint64_t drain;       // the issuer's last MMAs are complete
  uint32_t tmem_base;
  int bad_block;
  int abort;
};
static_assert(sizeof(TcBarriers) <= 256, "barrier block");

// ---------------------------------------------------------------- unit order

// Units of sequence s (rows of up to T tokens): prefill chunks of two or more
// rows (single rows are decode rows); in prefix mode any non-empty group with
// a non-empty shared prefix.
__device__ __forceinline__ int units_of(const TcParams& p, int s, int T, int* q_len, int* ctx) {
  const int q0 = p.cu_q_lens[s], q1 = p.cu_q_lens[s + 1];
  *q_len = q1 - q0;
  *ctx = p.context_lens[s];
  if (q0 < 0 || q1 > p.num_rows || q1 - q0 < (p.prefix_mode ? 1 : 2)) return 0;
  if (p.prefix_mode && *ctx <= 0) return 0;
  return (q1 - q0 + T - 1) / T;
}

// Units of sequence s that read at least V key tiles (every unit for V <= 1).
// Unit u's rows end at token f(u) = min((u + 1) T, q_len) - 1, position
// ctx - q_len + f(u), so it reads (ctx - q_len + f(u)) / 128 + 1 key tiles;
// f grows with u, so these units are the last ones of the sequence.
__device__ __forceinline__ int units_at_least(const TcParams& p, int s, int T, int V) {
  int q_len, ctx;
  const int U = units_of(p, s, T, &q_len, &ctx);
  if (U == 0 || V <= 1) return U;
  if (p.prefix_mode) return (ctx - 1) / kKeysTile + 1 >= V ? U : 0;
  // need min((u + 1) T, q_len) >= R
  const int64_t R = static_cast<int64_t>(kKeysTile) * (V - 1) + 1 - (static_cast<int64_t>(ctx) - q_len);
  if (R > q_len) return 0;
  const int64_t u_first = R <= T ? 0 : (R + T - 1) / T - 1;
  return U - static_cast<int>(u_first);
}

// Units of all sequences reading at least V key tiles, summed by one warp.
__device__ __forceinline__ int warp_count_at_least(const TcParams& p, int T, int V, int lane) {
  int c = 0;
  for (int s = lane; s < p.num_seqs; s += 32) c += units_at_least(p, s, T, V);
  return __reduce_add_sync(0xffffffffu, c);
}

// The unit of rank k (0-based) in the order of decreasing key-tile count
// (ties by sequence, then unit): its sequence and unit index, or false when
// there are at most k units. Computed by each warp on its own.
__device__ __forceinline__ bool unit_of_rank(const TcParams& p, int T, int k, int lane, int* s_out,
                                             int* u_out) {
  const int v_top = (p.max_blocks * kBlockSize - 1) / kKeysTile + 1;
  if (warp_count_at_least(p, T, 1, lane) <= k) return false;
  // largest V in [1, v_top] with more than k units reading at least V tiles
  int lo = 1, hi = v_top;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (warp_count_at_least(p, T, mid, lane) > k) lo = mid; else hi = mid - 1;
  }
  const int v = lo;
  const int above = v == v_top ? 0 : warp_count_at_least(p, T, v + 1, lane);
  int r = k - above;  // rank among the units whose count is v (>= v_top at the top)
  for (int base = 0; base < p.num_seqs; base += 32) {
    const int s = base + lane;
    int first = 0, e = 0;
    if (s < p.num_seqs) {
      int q_len, ctx;
      const int U = units_of(p, s, T, &q_len, &ctx);
      const int at = units_at_least(p, s, T, v);
      const int over = v == v_top ? 0 : units_at_least(p, s, T, v + 1);
      first = U - at;
      e = at - over;
    }
    int incl = e;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, e > 0 && incl - e <= r && r < incl);
    if (hit != 0) {
      const int src = __ffs(hit) - 1;
      *s_out = base + src;
      *u_out = __shfl_sync(0xffffffffu, first + (r - (incl - e)), src);
      return true;
    }
    r -= __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;  // not reached: the counts cover every unit
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h2);
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {

__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  TcBarriers& bar = *reinterpret_cast<TcBarriers*>(smem + kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  const int tq = kRowsTile / G;  // tokens per Q tile
  const int T = tq * p.q_tiles;  // tokens per unit
  // CTA rank k: unit rank k / hkv, KV head k % hkv, longest units first
  const int k_rank = static_cast<int>(blockIdx.x);
  const int g = k_rank % p.hkv;
  int s = 0, unit = 0;
  if (!unit_of_rank(p, T, k_rank / p.hkv, lane, &s, &unit)) return;
  const int q0 = p.cu_q_lens[s];
  const int q_len = p.cu_q_lens[s + 1] - q0;
  const int ctx = p.context_lens[s];
  const int tok0 = unit * T;
  const int ntok = min(T, q_len - tok0);          // tokens of this unit
  const int nq = (ntok + tq - 1) / tq;             // Q tiles with rows: 1 or 2
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
  const bool bad_len = p.prefix_mode ? (ctx % kBlockSize != 0 || ctx > p.max_blocks * kBlockSize)
                                     : (q_len > ctx || ctx > p.max_blocks * kBlockSize);
  if (bad_len) {
    if (tid == 0) status_or(p.d_status, PA_STATUS_BAD_LENGTH);
    for (int i = tid; i < ntok * G * kD; i += kThreadsTc) {
      const int tok = i / (G * kD), rem = i % (G * kD);
      const int64_t row = static_cast<int64_t>(q0 + tok0 + tok) * p.hq + g * G;
      if (p.prefix_mode) {
        p.pre_acc[row * kD + rem] = 0.f;
        if (rem % kD == 0) p.pre_ml[row + rem / kD] = make_float2(0.f, -1.f);  // poisoned partial
      } else {
        out[row * kD + rem] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }
  // Absolute position of the unit's first row; in prefix mode every row sits
  // past the whole prefix (a decode token after it) and sees all its keys.
  const int pos0 = p.prefix_mode ? ctx - 1 : ctx - q_len + tok0;
  const int max_pos = p.prefix_mode ? pos0 : pos0 + ntok - 1;  // last row's absolute position
  const int n_kt = max_pos / kKeysTile + 1;           // key tiles
  const int nblk = max_pos / kBlockSize + 1;          // pool blocks holding keys 0..max_pos

  if (tid == 0) {
    mbar_init(&bar.q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bar.k_full[i], 1);
      mbar_init(&bar.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bar.v_full[i], 1);
      mbar_init(&bar.v_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar.s_full[x], 1);
      mbar_init(&bar.p_full[x], 4);
      mbar_init(&bar.pv_done[x], 1);
    }
    mbar_init(&bar.drain, 1);
    bar.bad_block = 0;
    bar.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bar.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar.tmem_base;
  auto fail = [&]() {
    atomicOr(&bar.abort, 1);
    status_or(p.d_status, PA_STATUS_TIMEOUT);
  };

  // Block-table entries of key tile j, read as one batch of independent loads.
  auto tile_blocks = [&](int j, int (&ph)[kBlocksTile]) -> int {
    const int b0 = j * kBlocksTile;
    const int nb = min(kBlocksTile, nblk - b0);
    // prefix mode: the shared blocks are read through the group's first member
    const int64_t trow_idx = p.prefix_mode ? q0 : s;
    const int32_t* row = p.block_tables + trow_idx * p.max_blocks + b0;
#pragma unroll
    for (int b = 0; b < kBlocksTile; ++b) ph[b] = b < nb ? __ldg(row + b) : 0;
    return nb;
  };
  // One producer per operand: TMA of K tiles (warp 0) or V tiles (warp 10),
  // each 128 keys = 8 pool blocks x two 64-column halves. On leaving, it waits
  // (bounded) for the copies of the stages it filled last.
  auto produce = [&](const CUtensorMap* tm, int off, int stages, uint64_t* full, uint64_t* empty) {
    int ph[kBlocksTile], phn[kBlocksTile];
    int nb = tile_blocks(0, ph);
    int issued = 0;
    for (int j = 0; j < n_kt; ++j) {
      const int st = j % stages;
      const int nbn = j + 1 < n_kt ? tile_blocks(j + 1, phn) : 0;  // prefetch the next tile's table
      if (bar.abort != 0 || !mbar_wait_bounded(&empty[st], ((j / stages) & 1) ^ 1)) {
        if (bar.abort == 0) fail();
        break;
      }
      char* dst = smem + off + st * kTileBytes;
      mbar_arrive_expect_tx(&full[st], nb * 2 * (kBlockSize * 128));
      for (int b = 0; b < nb; ++b) {
        int phys = ph[b];
        if (phys < 0 || phys >= p.num_blocks) {  // keep the copy in bounds, zero the output
          bar.bad_block = 1;
          status_or(p.d_status, PA_STATUS_BAD_BLOCK);
          phys = 0;
        }
        const int row = phys * kBlockSize;
        tc::tma_load_3d(dst + b * (kBlockSize * 128), tm, 0, g, row, &full[st]);
        tc::tma_load_3d(dst + kHalf + b * (kBlockSize * 128), tm, 64, g, row, &full[st]);
      }
      issued = j + 1;
#pragma unroll
      for (int b = 0; b < kBlocksTile; ++b) ph[b] = phn[b];
      nb = nbn;
    }
    for (int j = max(0, issued - stages); j < issued; ++j)
      mbar_wait_bounded(&full[j % stages], (j / stages) & 1);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K loads
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      mbar_arrive_expect_tx(&bar.q_full, nq * 2 * kHalf);
      for (int x = 0; x < nq; ++x) {
        char* dq = smem + kOffQ + x * kTileBytes;
        tc::tma_load_3d(dq, &tm_q, 0, g * G, q0 + tok0 + x * tq, &bar.q_full);
        tc::tma_load_3d(dq + kHalf, &tm_q, 64, g * G, q0 + tok0 + x * tq, &bar.q_full);
      }
      produce(&tm_k, kOffK, kKStages, bar.k_full, bar.k_empty);
      mbar_wait_bounded(&bar.q_full, 0);
    }
  } else if (warp == kVWarp) {
    // ------------------------------------------------------------ V loads
    if (lane == 0) {
      tc::prefetch_tmap(&tm_v);
      produce(&tm_v, kOffV, kVStages, bar.v_full, bar.v_empty);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_bf16_f32(kRowsTile, kKeysTile, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(kRowsTile, kD, false, true);
      // No shared-memory load of the abort flag here: after an MMA commit the
      // next shared access of this thread holds up the tensor pipe's feed, so
      // the issuer learns of another role's abort through its own bounded
      // waits only.
      auto wait = [&](uint64_t* b, uint32_t parity) -> bool {
        if (!mbar_wait_bounded(b, parity)) return false;
        tc::fence_after_sync();
        return true;
      };
      // S_x = Q_x K_j^T into S_x's columns (K_j's stage is full)
      auto issue_s = [&](int x, int j) {
        const uint32_t sQ = smem_addr(smem + kOffQ + x * kTileBytes);
        const uint32_t sK = smem_addr(smem + kOffK + (j % kKStages) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t o = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + col_s(x), tc::smem_desc(sQ + o, 16, 1024),
                       tc::smem_desc(sK + o, 16, 1024), id_qk, kk > 0);
        }
        tc::mma_commit(&bar.s_full[x]);
      };
      // O_x += P_x V_j: key group kk (16 keys) is P columns 8 kk .. 8 kk + 7
      auto issue_pv = [&](int x, int j) {
        const uint32_t sV = smem_addr(smem + kOffV + (j % kVStages) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kKeysTile / 16; ++kk)
          tc::mma_bf16_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8,
                          tc::smem_desc(sV + kk * (16 * 128), kHalf, 1024), id_pv,
                          (j > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(&bar.pv_done[x]);
      };
      const bool two = nq == 2;
      bool ok = wait(&bar.q_full, 0) && wait(&bar.k_full[0], 0);
      if (ok) {
        issue_s(0, 0);
        if (two) issue_s(1, 0);
        tc::mma_commit(&bar.k_empty[0]);
      }
      for (int j = 0; ok && j < n_kt; ++j) {
        const bool next = j + 1 < n_kt;
        const int ks = (j + 1) % kKStages;
        ok = wait(&bar.v_full[j % kVStages], (j / kVStages) & 1) && wait(&bar.p_full[0], j & 1);
        if (!ok) break;
        issue_pv(0, j);
        // S_0(j+1) overwrites P_0(j), which the pipe reads first
        if (next) {
          if (!(ok = wait(&bar.k_full[ks], ((j + 1) / kKStages) & 1))) break;
          issue_s(0, j + 1);
        }
        if (two) {
          if (!(ok = wait(&bar.p_full[1], j & 1))) break;
          issue_pv(1, j);
        }
        tc::mma_commit(&bar.v_empty[j % kVStages]);
        if (next) {
          if (two) issue_s(1, j + 1);
          tc::mma_commit(&bar.k_empty[ks]);
        }
      }
      if (!ok && bar.abort == 0) fail();
      tc::mma_commit(&bar.drain);
      mbar_wait_bounded(&bar.drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // One thread per query row: warps 2-5 own Q tile 0, warps 6-9 Q tile 1.
    const int x = (warp - 2) >> 2;             // Q tile
    const int quad = warp & 3;                 // TMEM lane quarter this warp may access
    const int r = quad * 32 + lane;            // row within the Q tile
    const int ti = x * tq + r / G;             // token of the row within the unit
    const bool live = ti < ntok;
    const int pos = live ? pos0 + (p.prefix_mode ? 0 : x * tq + r / G) : -1;  // absolute position
    const int pos_first = p.prefix_mode ? pos0 : pos0 + x * tq;              // the tile's first row
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t scol = trow + col_s(x), ocol = trow + col_o(x);
    const float sl2 = p.scale_log2;
    // rows past the unit keep m = +inf: every weight is 0 and nothing moves
    float m = live ? -INFINITY : INFINITY, l = 0.f;
    bool ok = x < nq;
    // P = 2^(s - mm) of the 64 keys of half h of the tile (0 past the row's
    // position) into pk; returns their sum
    auto weights = [&](int h, float mm, bool full, int key0, uint32_t (&pk)[32]) -> float {
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
      uint32_t raw[2][32];
      tc::tmem_ld32(scol + h * 64, raw[0]);
      tc::tmem_ld32(scol + h * 64 + 32, raw[1]);
      tc::tmem_wait_ld();
      if (full) {
        const float2 c2 = make_float2(sl2, sl2);
        const float2 nm = make_float2(-mm, -mm);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 sv = make_float2(__uint_as_float(raw[c >> 4][(2 * c) & 31]),
                                        __uint_as_float(raw[c >> 4][(2 * c + 1) & 31]));
          const float2 t = __ffma2_rn(sv, c2, nm);
          const float2 w = make_float2(ex2(t.x), ex2(t.y));
          acc[c & 3] = __fadd2_rn(acc[c & 3], w);
          pk[c] = pack_bf16(w.x, w.y);
        }
      } else {
        // tiles that cross a row's position: keys past it get weight 0
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int key = key0 + h * 64 + 2 * c;
          const float a = key <= pos ? __uint_as_float(raw[c >> 4][(2 * c) & 31]) * sl2 : -INFINITY;
          const float b = key + 1 <= pos ? __uint_as_float(raw[c >> 4][(2 * c + 1) & 31]) * sl2 : -INFINITY;
          const float2 w = make_float2(a == -INFINITY ? 0.f : ex2(a - mm), b == -INFINITY ? 0.f : ex2(b - mm));
          acc[c & 3] = __fadd2_rn(acc[c & 3], w);
          pk[c] = pack_bf16(w.x, w.y);
        }
      }
      return ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
    };
    // the row's largest score among the tile's keys from column c0 on (0 or
    // 32; the columns before it hold P already) in the log2 domain, -inf if none
    auto row_max = [&](int key0, int c0) -> float {
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q * 32 < c0) continue;  // warp-uniform
        uint32_t raw[32];
        tc::tmem_ld32(scol + q * 32, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float v = key0 + q * 32 + e <= pos ? __uint_as_float(raw[e]) * sl2 : -INFINITY;
          mp[e & 7] = fmaxf(mp[e & 7], v);
        }
      }
      return fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
    };
    for (int j = 0; ok && j < n_kt; ++j) {
      ok = __all_sync(0xffffffffu, bar.abort == 0 && mbar_wait_bounded(&bar.s_full[x], j & 1));
      if (!ok) break;
      tc::fence_after_sync();
      const int key0 = j * kKeysTile;
      // every row of the tile sees every key of this tile: no mask
      const bool full = key0 + kKeysTile - 1 <= pos_first && sl2 > 0.f;
      float rs = 0.f, alpha = 1.f;
      bool warp_moved = false;
      // Each half's P goes to TMEM (keys 2c, 2c + 1 of the half in column
      // 32 h + c, over scores already read) as soon as it is final. P uses
      // the running max; a weight above 2^8 is possible only if the half's sum
      // is, and then the max of the scores still in TMEM is taken: for half 1
      // every key of half 0 is known to lie within 8 of the old max, so that
      // max decides. When it moves, half 0's stored P (half 1 only) is
      // rescaled in place and the half redone.
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
        float rh = weights(h, m, full, key0, pk);
        if (__any_sync(0xffffffffu, !(rh <= 256.f))) {
          const float mx = row_max(key0, h * 32);
          const bool need = mx > m + 8.f;
          if (__any_sync(0xffffffffu, need)) {
            warp_moved = true;
            const float mn = need ? mx : m;
            const float a = (m == -INFINITY) ? 0.f : (need ? ex2(m - mn) : 1.f);
            m = mn;
            alpha *= a;
            if (h == 1) {
              uint32_t p0[32];
              tc::tmem_wait_st();
              tc::tmem_ld32(scol, p0);
              tc::tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c)
                p0[c] = pack_bf16(__uint_as_float(p0[c] << 16) * a, __uint_as_float(p0[c] & 0xffff0000u) * a);
              tc::tmem_st32(scol, p0);
              rs *= a;
            }
            rh = weights(h, m, full, key0, pk);
          }
        }
        rs += rh;
        tc::tmem_st32(scol + h * 32, pk);
      }
      l = l * alpha + rs;
      // O holds key tiles 0 .. j-1 once P(j-1) V(j-1) is complete: rescale
      // this warp's rows only when a max moved
      if (j > 0 && warp_moved) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.pv_done[x], (j - 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(ocol + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st32(ocol + c * 32, o);
        }
      }
      tc::tmem_wait_st();
      // last tile: Q tile 0's rows zero the value rows no key of this unit may
      // use (thread r: key row r, both 64-column halves) before P_0 goes to
      // the MMA; P_1 V follows P_0 V in the pipe
      if (x == 0 && j == n_kt - 1) {
        const int vs = j % kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.v_full[vs], (j / kVStages) & 1));
        if (!ok) break;
        // rows past the context hold stale or poisoned slots; rows past the
        // last loaded block were never written by this CTA
        if (j * kKeysTile + r >= min(ctx, nblk * kBlockSize)) {
          char* sv = smem + kOffV + vs * kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(sv + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sv + kHalf + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full[x]);
    }
    if (ok && x < nq) {
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.pv_done[x], (n_kt - 1) & 1));
      if (ok) tc::fence_after_sync();
    }
    if (x < nq) {
      if (!ok) {
        if (lane == 0 && bar.abort == 0) fail();
      } else {
        // epilogue: this row's O from TMEM, 32 columns at a time
        const int rh = r % G;
        const int64_t idx = static_cast<int64_t>(q0 + tok0 + ti) * p.hq + g * G + rh;
        const float inv = (bar.bad_block || l == 0.f) ? 0.f : 1.f / l;
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(ocol + c * 32, o);
          tc::tmem_wait_ld();
          if (!live) continue;
          if (p.prefix_mode) {
            // the unnormalised partial (max m, sum l, accumulator) of this row
            float* arow = p.pre_acc + idx * kD + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(arow + e) =
                  make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                              __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
          } else {
            __nv_bfloat16* orow = out + idx * kD + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                w[q] = pack_bf16(__uint_as_float(o[e + 2 * q]) * inv, __uint_as_float(o[e + 2 * q + 1]) * inv);
              *reinterpret_cast<uint4*>(orow + e) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (live && p.prefix_mode) p.pre_ml[idx] = make_float2(m, bar.bad_block ? -1.f : l);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {

bool tc_supported(const PrefillArgs& a) {
  const int group = a.num_q_heads / a.pool.num_kv_heads;
  return a.pool.dtype == PA_BF16 && a.pool.head_dim == kD && kRowsTile % group == 0 &&
         group <= 8 && a.num_seqs <= kMaxPrefixSeqs && encode_tiled() != nullptr;
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  const int hkv = a.pool.num_kv_heads;
  const int group = a.num_q_heads / hkv;
  CUtensorMap tq, tk, tv;
  if (!make_tmap(&tq, a.q, kD, a.num_q_heads, a.num_tokens, 64, group, kRowsTile / group) ||
      !make_tmap(&tk, a.pool.k, kD, hkv, a.pool.num_blocks * kBlockSize, 64, 1, kBlockSize) ||
      !make_tmap(&tv, a.pool.v, kD, hkv, a.pool.num_blocks * kBlockSize, 64, 1, kBlockSize))
    return cudaErrorInvalidValue;
  if (a.num_seqs > kMaxPrefixSeqs) return cudaErrorInvalidValue;
  const int tq_tokens = kRowsTile / group;
  // Two Q tiles per unit share every K/V tile and overlap one tile's softmax
  // with the other's products, so a two-tile unit takes far less than twice a
  // one-tile unit; one-tile units win only when all of them fit on the SMs at
  // once.
  const int64_t pairs = (a.num_tokens + 2 * tq_tokens - 1) / (2 * tq_tokens);
  const int64_t budget = a.sm_budget > 0 ? a.sm_budget : device_sm_count();
  const int q_tiles = a.q_tiles == 1 || a.q_tiles == 2 ? a.q_tiles : (2 * pairs * hkv > budget ? 2 : 1);
  // at most sum(ceil(q_len / T)) <= num_tokens / T + (sequences with units):
  // every prefill chunk has two rows or more (prefix groups one or more)
  const int64_t with_units = a.prefix_mode ? a.num_seqs : std::min<int64_t>(a.num_seqs, a.num_tokens / 2);
  const int64_t units = (a.num_tokens + q_tiles * tq_tokens - 1) / (q_tiles * tq_tokens) + with_units;
  TcParams p;
  p.cu_q_lens = a.cu_q_lens;
  p.context_lens = a.context_lens;
  p.block_tables = a.block_tables;
  p.out = a.out;
  p.num_seqs = a.num_seqs;
  p.num_rows = a.num_tokens;
  p.hq = a.num_q_heads;
  p.hkv = hkv;
  p.group = group;
  p.max_blocks = a.max_blocks_per_seq;
  p.q_tiles = q_tiles;
  p.num_blocks = a.pool.num_blocks;
  p.scale_log2 = a.scale * kLog2e;
  p.d_status = a.d_status;
  p.prefix_mode = a.prefix_mode;
  p.pre_ml = static_cast<float2*>(a.pre_ml);
  p.pre_acc = static_cast<float*>(a.pre_acc);
  const int smem = kSmemTc;
  cudaError_t err =
      cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * hkv));  // an upper bound; the rest exit
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.beside_previous ? 1 : 0;
  err = cudaLaunchKernelEx(&cfg, prefill_tc_kernel, tq, tk, tv, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

bool prefix_supported(int dtype, int head_dim, int group, int num_groups) {
  return dtype == PA_BF16 && head_dim == kD && group >= 1 && group <= 8 && kRowsTile % group == 0 &&
         num_groups <= kMaxPrefixSeqs && encode_tiled() != nullptr;
}

cudaError_t launch_prefix_partials(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.num_tokens == 0) return cudaSuccess;
  if (!a.prefix_mode || a.pre_ml == nullptr || a.pre_acc == nullptr) return cudaErrorInvalidValue;
  return launch_prefill_tc(a, stream);
}

bool prefill_supported(int dtype, int head_dim, int group) {
  if (dtype != PA_F32 && dtype != PA_BF16) return false;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  return group == 1 || group == 2 || group == 4 || group == 8;
}

bool prefill_on_tensor_cores(const PrefillArgs& a) { return tc_supported(a); }

// bf16 with head_dim 128 runs on the tensor cores; the other shapes and fp32
// run on the CUDA-core kernel (prefill_simt.cu).
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0 || a.num_seqs == 0) return cudaSuccess;
  if (tc_supported(a)) return launch_prefill_tc(a, stream);
  return launch_prefill_simt(a, stream);
}

}  // namespace pa
