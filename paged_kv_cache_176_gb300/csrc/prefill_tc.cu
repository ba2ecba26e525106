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
// GB300 design (one CTA per 128 query rows of one KV head):
//  * The 128 rows are 128/G tokens x the G query heads that share the KV head,
//    so one K/V tile in shared memory serves the whole GQA group.
//  * Warp 0 moves Q once and then K tiles of 128 keys (8 pool blocks) into a
//    three-stage ring, warp 10 moves V tiles into a two-stage ring; each block
//    is one 3-D tiled TMA copy (64 head-dim columns x 16 tokens, 128-byte
//    swizzle) straight out of the paged pool, so the gather costs no extra pass.
//  * Warp 1 owns 512 TMEM columns and issues the MMAs from one thread:
//    S = Q K^T (128 x 128, fp32, double-buffered in TMEM) and, per key half,
//    O_h += P_h V_h with P_h read from TMEM (the A operand of a TS-MMA) and
//    V_h (64 keys x head_dim) from shared memory; tcgen05.commit signals
//    the mbarriers.
//  * Warps 2-9 hold two threads per query row, one per half of the key tile.
//    Each reads its 64 S columns from TMEM, applies the causal mask and the
//    online softmax in the log2 domain with its own (max, sum), writes P as
//    bf16 pairs back into the S columns it read, and rescales its own O_h only
//    when its max grows by more than 8 (lazy rescaling). Masked keys get
//    weight 0. The epilogue merges the two halves' (max, sum, O_h).
//  * On the last key tile each half zeroes the value rows of its own 64 keys
//    that lie past the context or past the loaded blocks, before it hands P_h
//    to the MMA that reads exactly those rows, so stale or NaN slots never
//    reach the result.
//  * Every wait is bounded; a timeout sets PA_STATUS_TIMEOUT and the CTA
//    leaves after releasing its TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace pa {
namespace {

constexpr int kD = 128;              // head_dim of the tensor-core path
constexpr int kRowsTile = 128;       // query rows per CTA (MMA M)
constexpr int kKeysTile = 128;       // keys per tile (MMA N of Q K^T)
constexpr int kBlocksTile = kKeysTile / kBlockSize;
constexpr int kThreadsTc = 352;      // warp 0 K loads, warp 1 MMA, warps 2-9 softmax, warp 10 V loads
constexpr int kVWarp = 10;
constexpr int kHalf = 16384;         // one 64-column half of a 128-row bf16 tile
constexpr int kTileBytes = 2 * kHalf;
constexpr int kKStages = 3;          // K is released as soon as S = Q K^T is done
constexpr int kVStages = 2;          // V is released after O += P V

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffP = kOffV + kVStages * kTileBytes;  // also holds the tile prefix at start-up
constexpr int kOffBar = kOffP + kTileBytes;
constexpr int kSmemTc = kOffBar + 256 + 1024;         // + barriers + alignment slack
constexpr int kMaxPrefixSeqs = kTileBytes / 4 - 1;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0;     // S buffers at 0 and 128
constexpr uint32_t kColO = 256;    // O accumulators: keys 0-63 of every tile at 256, keys 64-127 at 384

struct TcParams {
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  const int32_t* block_tables;
  void* out;
  int num_seqs, num_rows, hq, hkv, group, max_blocks;
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
  uint64_t s_full[2];
  uint64_t s_empty[2];
  uint64_t p_full[2][2];  // [S buffer][key half]: P of one 64-key half written
  uint64_t pv_done;
  uint32_t tmem_base;
  int bad_block;
  int abort;
};
static_assert(sizeof(TcBarriers) <= 256, "barrier block");

__device__ __forceinline__ int tc_tiles(const TcParams& p, int s, int tq) {
  const int q0 = p.cu_q_lens[s], q1 = p.cu_q_lens[s + 1];
  // prefill: chunks of two or more rows (single rows are decode rows);
  // prefix mode: any non-empty group with a non-empty shared prefix
  if (q0 < 0 || q1 > p.num_rows || q1 - q0 < (p.prefix_mode ? 1 : 2)) return 0;
  if (p.prefix_mode && p.context_lens[s] <= 0) return 0;
  return (q1 - q0 + tq - 1) / tq;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
  __shared__ int warp_sums[kThreadsTc / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  const int tq = kRowsTile / G;  // tokens per tile
  const int g = blockIdx.y;      // KV head

  // this CTA's (sequence, tile); tiles run from the last (longest) one down.
  // The prefix lives in the P buffer, which is free until the softmax starts.
  int* prefix = reinterpret_cast<int*>(smem + kOffP);
  block_exclusive_scan<kThreadsTc>(
      p.num_seqs, [&](int i) { return tc_tiles(p, i, tq); }, prefix, warp_sums);
  const int total = prefix[p.num_seqs];
  if (static_cast<int>(blockIdx.x) >= total) return;
  const int t_global = total - 1 - static_cast<int>(blockIdx.x);
  const int s = upper_index(prefix, p.num_seqs, t_global);
  const int tile = t_global - prefix[s];
  const int q0 = p.cu_q_lens[s];
  const int q_len = p.cu_q_lens[s + 1] - q0;
  const int ctx = p.context_lens[s];
  const int tok0 = tile * tq;
  const int ntok = min(tq, q_len - tok0);
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
  // Absolute position of the tile's first row; in prefix mode every row sits
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_empty[i], 8);
    }
    for (int b = 0; b < 2; ++b)
      for (int h = 0; h < 2; ++h) mbar_init(&bar.p_full[b][h], 4);
    mbar_init(&bar.pv_done, 1);
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
  // each 128 keys = 8 pool blocks x two 64-column halves.
  auto produce = [&](const CUtensorMap* tm, int off, int stages, uint64_t* full, uint64_t* empty) {
    int ph[kBlocksTile], phn[kBlocksTile];
    int nb = tile_blocks(0, ph);
    for (int j = 0; j < n_kt; ++j) {
      const int st = j % stages;
      const int nbn = j + 1 < n_kt ? tile_blocks(j + 1, phn) : 0;  // prefetch the next tile's table
      if (!mbar_wait_bounded(&empty[st], ((j / stages) & 1) ^ 1)) {
        atomicOr(&bar.abort, 1);
        return;
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
#pragma unroll
      for (int b = 0; b < kBlocksTile; ++b) ph[b] = phn[b];
      nb = nbn;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q and K loads
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      mbar_arrive_expect_tx(&bar.q_full, 2 * kHalf);
      tc::tma_load_3d(smem + kOffQ, &tm_q, 0, g * G, q0 + tok0, &bar.q_full);
      tc::tma_load_3d(smem + kOffQ + kHalf, &tm_q, 64, g * G, q0 + tok0, &bar.q_full);
      produce(&tm_k, kOffK, kKStages, bar.k_full, bar.k_empty);
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
      const uint32_t sQ = smem_addr(smem + kOffQ);
      const uint32_t sP = smem_addr(smem + kOffP);
      // S(j) = Q K_j^T into TMEM buffer j % 2; K_j's stage is free when it completes
      auto issue_s = [&](int j) -> bool {
        const int st = j % kKStages;
        if (!mbar_wait_bounded(&bar.k_full[st], (j / kKStages) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t sK = smem_addr(smem + kOffK + st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t o = (kk >> 2) * kHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + kColS0 + (j & 1) * kKeysTile, tc::smem_desc(sQ + o, 16, 1024),
                       tc::smem_desc(sK + o, 16, 1024), id_qk, kk > 0);
        }
        tc::mma_commit(&bar.s_full[j & 1]);
        tc::mma_commit(&bar.k_empty[st]);
        return true;
      };
      bool ok = mbar_wait_bounded(&bar.q_full, 0);
      if (ok) ok = issue_s(0);
      if (ok && n_kt > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int vs = j % kVStages;
        if (!mbar_wait_bounded(&bar.v_full[vs], (j / kVStages) & 1)) {
          ok = false;
          break;
        }
        const uint32_t sV = smem_addr(smem + kOffV + vs * kTileBytes);
        // O_h += P_h V_h for the two 64-key halves, each as soon as its P is
        // in TMEM (P_h sits in the first 32 columns of S_j's h-th half)
        for (int h = 0; h < 2 && ok; ++h) {
          // one barrier pair per S buffer: the next arrival on it needs
          // S(j + 2), which is issued only after this wait
          if (!mbar_wait_bounded(&bar.p_full[j & 1][h], (j >> 1) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t pcol = tmem + kColS0 + (j & 1) * kKeysTile + h * (kKeysTile / 2);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(tmem + kColO + h * kD, pcol + kk * 8,
                            tc::smem_desc(sV + (4 * h + kk) * (16 * 128), kHalf, 1024), id_pv,
                            (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (!ok) break;
        tc::mma_commit(&bar.v_empty[vs]);
        tc::mma_commit(&bar.pv_done);
        // S(j + 2) reuses S_j's columns: the tensor pipe runs it after P_j V_j
        if (j + 2 < n_kt && !issue_s(j + 2)) {
          ok = false;
          break;
        }
      }
      if (!ok) atomicOr(&bar.abort, 1);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Two threads per query row: half hf owns keys 64*hf .. 64*hf+63 of every
    // tile and runs its own online softmax into its own O accumulator; the
    // two (max, sum, O) triples are merged once, in the epilogue.
    const int quad = warp & 3;                 // TMEM lane quarter this warp may access
    const int hf = (warp - 2) >> 2;            // key half
    const int r = quad * 32 + lane;            // tile row owned by this thread
    const int ri = r / G;                      // token of the row within the tile
    const int pos = ri < ntok ? pos0 + (p.prefix_mode ? 0 : ri) : -1;  // absolute position (-1: padding row)
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t ocol = kColO + hf * kD;     // this half's O accumulator
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    constexpr int kCols = kKeysTile / 2;
    for (int j = 0; j < n_kt; ++j) {
      const int buf = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.s_full[buf], (j >> 1) & 1));
      if (!ok) break;
      tc::fence_after_sync();
      float sc[kCols];
      {
        uint32_t raw[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tc::tmem_ld32(trow + kColS0 + buf * kKeysTile + hf * kCols + c * 32, raw[c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) sc[c * 32 + e] = __uint_as_float(raw[c][e]);
      }
      // Key halves entirely below the diagonal need no mask (every key <=
      // every row's position); the others mask keys past each row's position.
      const int key0 = j * kKeysTile + hf * kCols;
      const bool full = key0 + kCols - 1 <= pos0 && p.scale_log2 > 0.f;
      float mx;
      {
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < kCols; ++c) mp[c & 7] = fmaxf(mp[c & 7], sc[c]);
        } else {
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            const float v = (key0 + c <= pos) ? sc[c] * p.scale_log2 : -INFINITY;
            sc[c] = v;
            mp[c & 7] = fmaxf(mp[c & 7], v);
          }
        }
        mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        if (full) mx *= p.scale_log2;  // scores in the log2 domain
      }
      // lazy running max: move it only when a score exceeds it by more than 8
      const bool need = mx > m + 8.f;
      const bool warp_need = __any_sync(0xffffffffu, need);
      const float mn = need ? mx : m;
      const float alpha = (m == -INFINITY) ? 0.f : (need ? ex2(m - mn) : 1.f);
      m = mn;
      // P = 2^(s - m) in registers (bf16 pairs) before touching shared P
      uint32_t pk[kCols / 2];
      float2 rsp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rsp[i] = make_float2(0.f, 0.f);
      if (full) {
        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm = make_float2(-m, -m);
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) {
          const float2 t = __ffma2_rn(make_float2(sc[2 * c], sc[2 * c + 1]), c2, nm);
          const float2 w = make_float2(ex2(t.x), ex2(t.y));
          rsp[c & 3] = __fadd2_rn(rsp[c & 3], w);
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(w.x, w.y);
          pk[c] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) {
          const float a = sc[2 * c], b = sc[2 * c + 1];
          const float2 w = make_float2(a == -INFINITY ? 0.f : ex2(a - m), b == -INFINITY ? 0.f : ex2(b - m));
          rsp[c & 3] = __fadd2_rn(rsp[c & 3], w);
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(w.x, w.y);
          pk[c] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      const float rs = ((rsp[0].x + rsp[0].y) + (rsp[1].x + rsp[1].y)) +
                       ((rsp[2].x + rsp[2].y) + (rsp[3].x + rsp[3].y));
      l = l * alpha + rs;
      // O_hf holds tiles 0 .. j-1 once P_{j-1} V_{j-1} is complete: rescale
      // this warp's rows only when its running max moved
      if (j > 0 && warp_need) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.pv_done, (j - 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(trow + ocol + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st32(trow + ocol + c * 32, o);
        }
      }
      // P (bf16 pairs) over the first 32 columns of this half's S columns
      tc::tmem_st32(trow + kColS0 + buf * kKeysTile + hf * kCols, pk);
      tc::tmem_wait_st();
      // last tile: zero the value rows no key of this CTA may use. O_h += P_h V_h
      // reads keys 64*hf .. 64*hf+63 over all head_dim columns, so the 128
      // threads of this half clear exactly those rows (thread r: key
      // 64*hf + r/2, head_dim columns 64*(r&1) .. +63) before they arrive
      // on p_full[buf][hf].
      if (j == n_kt - 1) {
        const int vs = j % kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.v_full[vs], (j / kVStages) & 1));
        if (!ok) break;
        // rows past the context hold stale or poisoned slots; rows past the
        // last loaded block were never written by this CTA
        const int kr = hf * (kKeysTile / 2) + (r >> 1);
        if (j * kKeysTile + kr >= min(ctx, nblk * kBlockSize)) {
          char* sv = smem + kOffV + vs * kTileBytes + (r & 1) * kHalf;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sv + kr * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full[buf][hf]);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar.pv_done, (n_kt - 1) & 1));
      if (ok) tc::fence_after_sync();
    }
    if (!ok) atomicOr(&bar.abort, 1);
    // this half's (max, sum) for the epilogue merge; the P tile is free now
    float* ml = reinterpret_cast<float*>(smem + kOffP);
    ml[(hf * kRowsTile + r) * 2] = m;
    ml[(hf * kRowsTile + r) * 2 + 1] = l;
  }

  __syncthreads();  // every role done issuing; the last P.V is complete
  if (warp >= 2 && warp < kVWarp) {
    const int quad = warp & 3;
    const int hf = (warp - 2) >> 2;  // this thread writes head_dim columns 64*hf .. 64*hf+63
    const int r = quad * 32 + lane;
    const int ri = r / G, rh = r % G;
    if (bar.abort == 0) {
      // epilogue: merge the two key halves, O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1)
      const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      uint32_t raw[2][2][32];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 2; ++c) tc::tmem_ld32(trow + kColO + h * kD + hf * 64 + c * 32, raw[h][c]);
      tc::tmem_wait_ld();
      if (ri < ntok) {
        const float* ml = reinterpret_cast<const float*>(smem + kOffP);
        const float m0 = ml[r * 2], l0 = ml[r * 2 + 1];
        const float m1 = ml[(kRowsTile + r) * 2], l1 = ml[(kRowsTile + r) * 2 + 1];
        const float mm = fmaxf(m0, m1);
        const float a0 = m0 == -INFINITY ? 0.f : ex2(m0 - mm);
        const float a1 = m1 == -INFINITY ? 0.f : ex2(m1 - mm);
        if (p.prefix_mode) {
          // the unnormalised partial (max mm, sum, accumulator) of this row
          const int64_t idx = static_cast<int64_t>(q0 + tok0 + ri) * p.hq + g * G + rh;
          float* arow = p.pre_acc + idx * kD + hf * 64;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float x[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                x[k] = __uint_as_float(raw[0][c][e + k]) * a0 + __uint_as_float(raw[1][c][e + k]) * a1;
              *reinterpret_cast<float4*>(arow + c * 32 + e) = make_float4(x[0], x[1], x[2], x[3]);
            }
          if (hf == 0) p.pre_ml[idx] = make_float2(mm, bar.bad_block ? -1.f : a0 * l0 + a1 * l1);
        } else {
        const float inv = bar.bad_block ? 0.f : 1.f / (a0 * l0 + a1 * l1);
        const float s0 = a0 * inv, s1 = a1 * inv;
        __nv_bfloat16* orow =
            out + (static_cast<int64_t>(q0 + tok0 + ri) * p.hq + g * G + rh) * kD + hf * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i0 = e + 2 * k;
              const float x0 = __uint_as_float(raw[0][c][i0]) * s0 + __uint_as_float(raw[1][c][i0]) * s1;
              const float x1 = __uint_as_float(raw[0][c][i0 + 1]) * s0 + __uint_as_float(raw[1][c][i0 + 1]) * s1;
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
              w[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    } else if (r == 0 && hf == 0) {
      status_or(p.d_status, PA_STATUS_TIMEOUT);
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
  p.num_blocks = a.pool.num_blocks;
  p.scale_log2 = a.scale * kLog2e;
  p.d_status = a.d_status;
  p.prefix_mode = a.prefix_mode;
  p.pre_ml = static_cast<float2*>(a.pre_ml);
  p.pre_acc = static_cast<float*>(a.pre_acc);
  const int tq_tokens = kRowsTile / group;
  const int tiles = (a.num_tokens + tq_tokens - 1) / tq_tokens + a.num_seqs;  // upper bound
  const int smem = kSmemTc;
  if (a.num_seqs > kMaxPrefixSeqs) return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, hkv);
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
