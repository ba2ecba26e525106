// decode.cu -- paged decode attention on sm_103a (SIMT, HBM-bound).
//
// What it computes: for every decode sequence s and query head h (KV head
// g = h / G), o[s,h] = softmax_p(scale * q[s,h] . K_s[p,g]) V_s[p,g] over
// p < ctx_s, where K_s/V_s is the sequence's cache gathered through its block
// table. The block loop is the paged_attn pseudo-kernel of "Inference engine
// core techniques", section 1.4 (per page: look up the physical page, read
// its K/V, accumulate with an online softmax); the gather is K_r =
// gather(K_pool, table_r) from the "C13 L2 serving" page.
//
// GB300 design:
//  * Persistent grid, one CTA per SM. The blocks of all decode sequences,
//    concatenated in sequence order, are cut into `grid` equal contiguous
//    ranges, one per CTA (balanced split-K: every CTA reads the same number of
//    KV bytes whatever the context mix). A sequence inside one CTA's range is
//    finished by that CTA; a sequence that straddles CTAs leaves one partial
//    (max, sum, accumulator) per CTA, merged by decode_reduce_kernel. The cut
//    depends only on the context lengths, so the result is bit-identical under
//    any relabelling of physical blocks or sharing of blocks.
//  * A pool block stores its 16 tokens x all KV heads contiguously, so one
//    1-D bulk copy (cp.async.bulk) moves a whole block of K (and one of V)
//    into shared memory: 16-byte aligned, fully coalesced, no per-thread
//    address math. A 3-4 stage mbarrier pipeline keeps >= 2 blocks (up to
//    128 KB) in flight per SM. The block table is read once per block for all
//    heads.
//  * Warp w serves KV head w % Hkv; its G query heads live in registers, so
//    each K/V element read from shared memory feeds G FMAs (GQA grouping).
//    Lanes split a token's head_dim in 16-byte chunks; a warp works on several
//    tokens at once; packed fp32x2 FMAs (FFMA2) do the dot products and the
//    P.V update.
//  * Online softmax in the log2 domain (q pre-scaled by scale*log2 e) with a
//    lazy running max: the accumulator is rescaled only when a new score
//    exceeds the running max by more than 8 (factor 256), which keeps every
//    weight <= 256 and skips almost all rescales.
//  * Tokens past the context (the tail of a last block) are never loaded and
//    never touched, so stale or NaN slots cannot leak into the result.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxDecodeCtas = 1024;  // workspace is sized for this many partial slots
constexpr int kTokBatch = 4;          // tokens per softmax update per token group
constexpr float kRescaleThreshold = 8.0f;

template <typename T, int D, int G>
struct Cfg {
  static constexpr int kElt = sizeof(T);
  static constexpr int kVec = 16 / kElt;                      // elements per 16-byte chunk
  static constexpr int kC = (64 / G < D / 8) ? 64 / G : D / 8;  // elements per lane per token
  static constexpr int kLpt = D / kC;                         // lanes per token
  static constexpr int kTg = 32 / kLpt;                       // tokens per warp step
  static constexpr int kChunks = kC / kVec;                   // chunks per lane per token
  static constexpr int kPairs = kC / 2;
  static_assert(kC % kVec == 0, "lane slice must be whole 16-byte chunks");
  static_assert(kLpt >= 1 && kLpt <= 32 && 32 % kLpt == 0, "bad lane split");
};

struct SmemLayout {
  int stages;
  int tokens_per_unit;  // tokens of one block moved per pipeline stage (16, 8 or 4)
  int parts;            // 16 / tokens_per_unit
  int part_bytes;       // one K (or V) part: tokens_per_unit * Hkv * D * elt
  int off_bars, off_flags, off_merge, off_prefix, total;
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }
inline size_t align_up_sz(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout make_layout(int stages, int tokens_per_unit, int hkv, int d,
                                                  int elt, int wh, int group, int num_seqs) {
  SmemLayout L;
  L.stages = stages;
  L.tokens_per_unit = tokens_per_unit;
  L.parts = kBlockSize / tokens_per_unit;
  L.part_bytes = tokens_per_unit * hkv * d * elt;
  int off = stages * 2 * L.part_bytes;
  L.off_bars = align_up(off, 16);
  L.off_flags = L.off_bars + stages * 8;
  L.off_merge = align_up(L.off_flags + stages * 4, 16);
  const int merge_bytes = (wh - 1) * hkv * group * (d + 2) * 4;
  L.off_prefix = align_up(L.off_merge + merge_bytes, 16);
  L.total = align_up(L.off_prefix + (num_seqs + 1) * 4, 128);
  return L;
}

struct DecodeParams {
  const char* k_pool;
  const char* v_pool;
  int64_t num_blocks;
  int hkv;
  int hq;
  int wh;  // warps per KV head
  const void* q;
  void* out;
  const int32_t* cu_q_lens;
  int num_seqs;
  int num_rows;  // rows of q/out
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* context_lens;
  float scale_log2;
  int* ws_prefix;  // [num_seqs + 1]
  float2* ws_ml;   // [slots, hq] (m, l)
  float* ws_acc;   // [slots, hq, D]
  int* d_status;
  SmemLayout L;
};

// Blocks the decode kernel reads for sequence s (0 when s is not a decode
// sequence or its lengths are invalid).
__device__ __forceinline__ int decode_blocks(const DecodeParams& p, int s, bool* bad) {
  int q_len = 1;
  if (p.cu_q_lens != nullptr) {
    q_len = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
    if (q_len < 0 || p.cu_q_lens[s] < 0 || p.cu_q_lens[s + 1] > p.num_rows) {
      *bad = true;  // malformed cu_q_lens: never index q/out with it
      return 0;
    }
  }
  if (q_len != 1) return 0;
  const int ctx = p.context_lens[s];
  if (ctx < 1 || ctx > p.max_blocks * kBlockSize) {
    *bad = true;
    return 0;
  }
  return (ctx + kBlockSize - 1) / kBlockSize;
}

__device__ __forceinline__ int query_row(const DecodeParams& p, int s) {
  return p.cu_q_lens != nullptr ? p.cu_q_lens[s] : s;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  using C = Cfg<T, D, G>;
  extern __shared__ __align__(128) char smem[];
  const SmemLayout& L = p.L;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
  int* flags = reinterpret_cast<int*>(smem + L.off_flags);
  float* merge = reinterpret_cast<float*>(smem + L.off_merge);
  int* prefix = reinterpret_cast<int*>(smem + L.off_prefix);
  __shared__ int warp_sums[kWarps];
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int S = p.num_seqs;

  if (tid == 0) {
    for (int i = 0; i < L.stages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  bool bad_len = false;
  block_exclusive_scan<kThreads>(
      S, [&](int s) { return decode_blocks(p, s, &bad_len); }, prefix, warp_sums);
  if (bad_len && blockIdx.x == 0) status_or(p.d_status, PA_STATUS_BAD_LENGTH);

  // Invalid decode sequences (bad lengths) get zero output rows, written once.
  if (blockIdx.x == 0) {
    for (int s = warp; s < S; s += kWarps) {
      bool bad = false;
      const bool decode_row = decode_blocks(p, s, &bad) > 0 || bad;
      int q_len = 1;
      if (p.cu_q_lens != nullptr) q_len = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
      const int row = query_row(p, s);
      if (decode_row && bad && q_len == 1 && row >= 0 && row < p.num_rows) {
        T* o = static_cast<T*>(p.out) + static_cast<int64_t>(query_row(p, s)) * p.hq * D;
        for (int i = lane; i < p.hq * D; i += 32) o[i] = from_float<T>(0.f);
      }
    }
    for (int i = tid; i <= S; i += kThreads) p.ws_prefix[i] = prefix[i];
  }

  const int64_t B = prefix[S];
  const int64_t grid = gridDim.x;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * B / grid;
  const int64_t hi = (static_cast<int64_t>(blockIdx.x) + 1) * B / grid;
  if (lo >= hi) return;

  const int parts = L.parts;
  const int tpu = L.tokens_per_unit;
  const int64_t n_units = (hi - lo) * parts;
  const int token_bytes = p.hkv * D * C::kElt;

  // ---------------------------------------------------------------- producer
  // Thread 0 issues the bulk copies, running `stages` units ahead.
  int prod_seq = upper_index(prefix, S, lo);
  auto issue = [&](int64_t u) {
    const int st = static_cast<int>(u % L.stages);
    const int64_t blk = lo + u / parts;
    const int part = static_cast<int>(u % parts);
    while (prefix[prod_seq + 1] <= blk) ++prod_seq;
    const int s = prod_seq;
    const int j = static_cast<int>(blk - prefix[s]);  // logical block of sequence s
    const int ctx = p.context_lens[s];
    const int phys = p.block_tables[static_cast<int64_t>(s) * p.max_blocks + j];
    const int first_tok = j * kBlockSize + part * tpu;
    const int ntok = min(tpu, ctx - first_tok);
    if (phys < 0 || phys >= p.num_blocks) {
      flags[st] = -1;
      status_or(p.d_status, PA_STATUS_BAD_BLOCK);
      mbar_arrive(&bars[st]);
    } else if (ntok <= 0) {
      flags[st] = 0;
      mbar_arrive(&bars[st]);
    } else {
      flags[st] = ntok;
      const uint32_t bytes = static_cast<uint32_t>(ntok * token_bytes);
      const int64_t src = (static_cast<int64_t>(phys) * kBlockSize + part * tpu) * token_bytes;
      char* kdst = smem + st * 2 * L.part_bytes;
      mbar_arrive_expect_tx(&bars[st], 2 * bytes);
      bulk_g2s(kdst, p.k_pool + src, bytes, &bars[st]);
      bulk_g2s(kdst + L.part_bytes, p.v_pool + src, bytes, &bars[st]);
    }
  };
  if (tid == 0) {
    for (int64_t u = 0; u < min(static_cast<int64_t>(L.stages), n_units); ++u) issue(u);
  }

  // ---------------------------------------------------------------- consumers
  const int g = warp % p.hkv;       // this warp's KV head
  const int sub = warp / p.hkv;     // which share of a unit's tokens
  const bool active = warp < p.hkv * p.wh;
  const int tg = lane / C::kLpt;    // token slot within a warp step
  const int kl = lane % C::kLpt;    // 16-byte chunk column
  const int tok_stride = p.wh * C::kTg;

  float2 qf[G][C::kPairs];
  float2 acc[G][C::kPairs];
  float m[G], l[G];

  int64_t u = 0;
  int s = upper_index(prefix, S, lo);
  while (u < n_units) {
    while (prefix[s + 1] <= lo + u / parts) ++s;
    const int64_t seq_lo = max(lo, static_cast<int64_t>(prefix[s]));
    const int64_t seq_hi = min(hi, static_cast<int64_t>(prefix[s + 1]));
    const int64_t seq_units = (seq_hi - seq_lo) * parts;
    const bool whole = prefix[s] >= lo && prefix[s + 1] <= hi;
    const int row = query_row(p, s);
    const int ctx = p.context_lens[s];

    // load this warp's G query heads (pre-scaled into the log2 domain)
    if (active) {
      const T* qrow = static_cast<const T*>(p.q) + (static_cast<int64_t>(row) * p.hq + g * G) * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          const int dim0 = (kl + C::kLpt * c) * C::kVec;
          const uint4 raw = *reinterpret_cast<const uint4*>(qrow + h * D + dim0);
          float vals[C::kVec];
          if constexpr (sizeof(T) == 2) {
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = bf16x2_to_float2(w[i]);
              vals[2 * i] = f.x;
              vals[2 * i + 1] = f.y;
            }
          } else {
            vals[0] = __uint_as_float(raw.x);
            vals[1] = __uint_as_float(raw.y);
            vals[2] = __uint_as_float(raw.z);
            vals[3] = __uint_as_float(raw.w);
          }
#pragma unroll
          for (int i = 0; i < C::kVec / 2; ++i)
            qf[h][c * (C::kVec / 2) + i] =
                make_float2(vals[2 * i] * p.scale_log2, vals[2 * i + 1] * p.scale_log2);
        }
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < C::kPairs; ++i) acc[h][i] = make_float2(0.f, 0.f);
      }
    }
    bool poisoned = false;

    for (int64_t su = 0; su < seq_units; ++su, ++u) {
      const int st = static_cast<int>(u % L.stages);
      const uint32_t parity = static_cast<uint32_t>((u / L.stages) & 1);
      // every lane waits; the warp goes on only if all its lanes saw the data
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], parity));
      if (!ok) abort_flag = 1;
      const int ntok = flags[st];
      if (ntok < 0) poisoned = true;
      if (active && ntok > 0 && ok) {
        const T* kbase = reinterpret_cast<const T*>(smem + st * 2 * L.part_bytes);
        const T* vbase = reinterpret_cast<const T*>(smem + st * 2 * L.part_bytes + L.part_bytes);
        for (int t0 = sub * C::kTg; t0 < tpu; t0 += tok_stride * kTokBatch) {
          float sc[kTokBatch][G];
          bool valid[kTokBatch];
#pragma unroll
          for (int b = 0; b < kTokBatch; ++b) {
            const int t = t0 + b * tok_stride + tg;
            valid[b] = t < ntok;
            float2 part[G];
#pragma unroll
            for (int h = 0; h < G; ++h) part[h] = make_float2(0.f, 0.f);
            if (valid[b]) {
              const T* krow = kbase + (t * p.hkv + g) * D;
#pragma unroll
              for (int c = 0; c < C::kChunks; ++c) {
                const uint4 raw =
                    *reinterpret_cast<const uint4*>(krow + (kl + C::kLpt * c) * C::kVec);
                float2 kf[C::kVec / 2];
                if constexpr (sizeof(T) == 2) {
                  kf[0] = bf16x2_to_float2(raw.x);
                  kf[1] = bf16x2_to_float2(raw.y);
                  kf[2] = bf16x2_to_float2(raw.z);
                  kf[3] = bf16x2_to_float2(raw.w);
                } else {
                  kf[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
                  kf[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
                }
#pragma unroll
                for (int i = 0; i < C::kVec / 2; ++i)
#pragma unroll
                  for (int h = 0; h < G; ++h)
                    part[h] = __ffma2_rn(qf[h][c * (C::kVec / 2) + i], kf[i], part[h]);
              }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) sc[b][h] = part[h].x + part[h].y;
          }
          // complete the dot products across the lanes sharing a token
#pragma unroll
          for (int off = C::kLpt / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int b = 0; b < kTokBatch; ++b)
#pragma unroll
              for (int h = 0; h < G; ++h) sc[b][h] += __shfl_xor_sync(0xffffffffu, sc[b][h], off);
          // online softmax update (lazy max)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float mx = -INFINITY;
#pragma unroll
            for (int b = 0; b < kTokBatch; ++b)
              if (valid[b]) mx = fmaxf(mx, sc[b][h]);
            if (mx > m[h] + kRescaleThreshold) {
              const float a = exp2f(m[h] - mx);  // 0 when m = -inf
              l[h] *= a;
#pragma unroll
              for (int i = 0; i < C::kPairs; ++i) acc[h][i] = make_float2(acc[h][i].x * a, acc[h][i].y * a);
              m[h] = mx;
            }
#pragma unroll
            for (int b = 0; b < kTokBatch; ++b) {
              const float w = valid[b] ? exp2f(sc[b][h] - m[h]) : 0.f;
              sc[b][h] = w;
              l[h] += w;
            }
          }
          // P.V
#pragma unroll
          for (int b = 0; b < kTokBatch; ++b) {
            if (!valid[b]) continue;
            const int t = t0 + b * tok_stride + tg;
            const T* vrow = vbase + (t * p.hkv + g) * D;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              const uint4 raw = *reinterpret_cast<const uint4*>(vrow + (kl + C::kLpt * c) * C::kVec);
              float2 vf[C::kVec / 2];
              if constexpr (sizeof(T) == 2) {
                vf[0] = bf16x2_to_float2(raw.x);
                vf[1] = bf16x2_to_float2(raw.y);
                vf[2] = bf16x2_to_float2(raw.z);
                vf[3] = bf16x2_to_float2(raw.w);
              } else {
                vf[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
                vf[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
              }
#pragma unroll
              for (int h = 0; h < G; ++h) {
                const float2 w2 = make_float2(sc[b][h], sc[b][h]);
#pragma unroll
                for (int i = 0; i < C::kVec / 2; ++i)
                  acc[h][c * (C::kVec / 2) + i] = __ffma2_rn(w2, vf[i], acc[h][c * (C::kVec / 2) + i]);
              }
            }
          }
        }
      }
      __syncthreads();  // stage st fully consumed
      if (abort_flag) break;
      if (tid == 0 && u + L.stages < n_units) issue(u + L.stages);
    }
    if (abort_flag) {
      if (tid == 0) status_or(p.d_status, PA_STATUS_TIMEOUT);
      return;
    }

    // ------------------------------------------------------------ finish s
    // 1. merge the token slots of each warp (lanes with equal kl)
    if (active) {
#pragma unroll
      for (int off = C::kLpt; off < 32; off <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
          const float lo_ = __shfl_xor_sync(0xffffffffu, l[h], off);
          const float mn = fmaxf(m[h], mo);
          const float a = (m[h] == -INFINITY) ? 0.f : exp2f(m[h] - mn);
          const float b = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
          l[h] = l[h] * a + lo_ * b;
#pragma unroll
          for (int i = 0; i < C::kPairs; ++i) {
            const float ox = __shfl_xor_sync(0xffffffffu, acc[h][i].x, off);
            const float oy = __shfl_xor_sync(0xffffffffu, acc[h][i].y, off);
            acc[h][i] = make_float2(acc[h][i].x * a + ox * b, acc[h][i].y * a + oy * b);
          }
          m[h] = mn;
        }
      }
    }
    // 2. merge the warps that share a KV head through shared memory
    if (p.wh > 1) {
      if (active && sub > 0 && tg == 0) {
        float* slot = merge + ((sub - 1) * p.hkv + g) * G * (D + 2);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float* hs = slot + h * (D + 2);
          if (kl == 0) {
            hs[D] = m[h];
            hs[D + 1] = l[h];
          }
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
            for (int i = 0; i < C::kVec / 2; ++i) {
              const int dim = (kl + C::kLpt * c) * C::kVec + 2 * i;
              hs[dim] = acc[h][c * (C::kVec / 2) + i].x;
              hs[dim + 1] = acc[h][c * (C::kVec / 2) + i].y;
            }
        }
      }
      __syncthreads();
      if (active && sub == 0) {
        for (int w2 = 1; w2 < p.wh; ++w2) {
          const float* slot = merge + ((w2 - 1) * p.hkv + g) * G * (D + 2);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float* hs = slot + h * (D + 2);
            const float mo = hs[D], lo_ = hs[D + 1];
            const float mn = fmaxf(m[h], mo);
            const float a = (m[h] == -INFINITY) ? 0.f : exp2f(m[h] - mn);
            const float b = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
            l[h] = l[h] * a + lo_ * b;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
              for (int i = 0; i < C::kVec / 2; ++i) {
                const int dim = (kl + C::kLpt * c) * C::kVec + 2 * i;
                float2& r = acc[h][c * (C::kVec / 2) + i];
                r = make_float2(r.x * a + hs[dim] * b, r.y * a + hs[dim + 1] * b);
              }
            m[h] = mn;
          }
        }
      }
      __syncthreads();  // merge buffer free for the next sequence
    }
    // 3. write: the final row when this CTA saw the whole sequence, else a partial
    if (active && sub == 0 && tg == 0) {
      if (whole) {
        T* orow = static_cast<T*>(p.out) + (static_cast<int64_t>(row) * p.hq + g * G) * D;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float inv = poisoned ? 0.f : 1.f / l[h];
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            const int dim0 = (kl + C::kLpt * c) * C::kVec;
            if constexpr (sizeof(T) == 2) {
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 r = acc[h][c * 4 + i];
                const __nv_bfloat162 bb = __floats2bfloat162_rn(r.x * inv, r.y * inv);
                w[i] = *reinterpret_cast<const uint32_t*>(&bb);
              }
              *reinterpret_cast<uint4*>(orow + h * D + dim0) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              const float2 r0 = acc[h][c * 2], r1 = acc[h][c * 2 + 1];
              *reinterpret_cast<float4*>(orow + h * D + dim0) =
                  make_float4(r0.x * inv, r0.y * inv, r1.x * inv, r1.y * inv);
            }
          }
        }
      } else {
        const int64_t slot = static_cast<int64_t>(blockIdx.x) + s;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const int hh = g * G + h;
          if (kl == 0) p.ws_ml[slot * p.hq + hh] = make_float2(m[h], poisoned ? -1.f : l[h]);
          float* arow = p.ws_acc + (slot * p.hq + hh) * D;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) {
            const int dim0 = (kl + C::kLpt * c) * C::kVec;
#pragma unroll
            for (int i = 0; i < C::kVec / 4; ++i) {
              const float2 r0 = acc[h][c * (C::kVec / 2) + 2 * i];
              const float2 r1 = acc[h][c * (C::kVec / 2) + 2 * i + 1];
              *reinterpret_cast<float4*>(arow + dim0 + 4 * i) = make_float4(r0.x, r0.y, r1.x, r1.y);
            }
          }
        }
      }
    }
  }
  pdl_launch_dependents();
}

// Merge the partials of sequences that straddle CTAs: o = sum_c a_c acc_c /
// sum_c a_c l_c with a_c = 2^(m_c - max_c m_c).
template <typename T, int D>
__global__ void __launch_bounds__(256) decode_reduce_kernel(const DecodeParams p, int grid) {
  pdl_wait_primary();
  const int s = blockIdx.x;
  const int* prefix = p.ws_prefix;
  const int64_t B = prefix[p.num_seqs];
  const int64_t a0 = prefix[s], a1 = prefix[s + 1];
  if (a1 <= a0) return;
  // CTA c covers blocks [c*B/grid, (c+1)*B/grid)
  const int64_t c_first = ((a0 + 1) * grid - 1) / B;
  const int64_t c_last = (a1 * grid - 1) / B;
  if (c_first == c_last) return;  // finished by the decode kernel
  const int row = query_row(p, s);
  T* orow = static_cast<T*>(p.out) + static_cast<int64_t>(row) * p.hq * D;
  for (int idx = threadIdx.x; idx < p.hq * (D / 4); idx += blockDim.x) {
    const int h = idx / (D / 4);
    const int e = (idx % (D / 4)) * 4;
    float mx = -INFINITY;
    bool poisoned = false;
    for (int64_t c = c_first; c <= c_last; ++c) {
      if (c * B / grid == (c + 1) * B / grid) continue;  // CTA with an empty range
      const float2 ml = p.ws_ml[(c + s) * p.hq + h];
      mx = fmaxf(mx, ml.x);
      poisoned |= ml.y < 0.f;
    }
    float lsum = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t c = c_first; c <= c_last; ++c) {
      if (c * B / grid == (c + 1) * B / grid) continue;
      const float2 ml = p.ws_ml[(c + s) * p.hq + h];
      const float a = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - mx);
      lsum += a * ml.y;
      const float4 v = *reinterpret_cast<const float4*>(p.ws_acc + ((c + s) * p.hq + h) * D + e);
      o.x += a * v.x;
      o.y += a * v.y;
      o.z += a * v.z;
      o.w += a * v.w;
    }
    const float inv = poisoned ? 0.f : 1.f / lsum;
    T* dst = orow + h * D + e;
    dst[0] = from_float<T>(o.x * inv);
    dst[1] = from_float<T>(o.y * inv);
    dst[2] = from_float<T>(o.z * inv);
    dst[3] = from_float<T>(o.w * inv);
  }
}

template <typename T, int D, int G>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  const int hkv = a.pool.num_kv_heads;
  const int wh = kWarps / hkv;
  const int elt = sizeof(T);
  const int token_bytes = hkv * D * elt;
  // tokens of one block moved per stage: whole blocks when a K+V block fits 64 KB
  int tpu = kBlockSize;
  while (tpu > 4 && 2 * tpu * token_bytes > 64 * 1024) tpu /= 2;
  const int smem_limit = 227 * 1024 - 1024;  // leave room for static shared memory
  SmemLayout L = make_layout(4, tpu, hkv, D, elt, wh, G, a.num_seqs);
  if (L.total > smem_limit) L = make_layout(3, tpu, hkv, D, elt, wh, G, a.num_seqs);
  if (L.total > smem_limit) L = make_layout(2, tpu, hkv, D, elt, wh, G, a.num_seqs);
  if (L.total > smem_limit) return cudaErrorInvalidValue;

  int grid = a.grid_override > 0 ? a.grid_override : device_sm_count();
  grid = std::min(grid, kMaxDecodeCtas);

  DecodeParams p;
  p.k_pool = static_cast<const char*>(a.pool.k);
  p.v_pool = static_cast<const char*>(a.pool.v);
  p.num_blocks = a.pool.num_blocks;
  p.hkv = hkv;
  p.hq = a.num_q_heads;
  p.wh = wh;
  p.q = a.q;
  p.out = a.out;
  p.cu_q_lens = a.cu_q_lens;
  p.num_seqs = a.num_seqs;
  p.num_rows = a.num_rows;
  p.block_tables = a.block_tables;
  p.max_blocks = a.max_blocks_per_seq;
  p.context_lens = a.context_lens;
  p.scale_log2 = a.scale * kLog2e;
  char* ws = static_cast<char*>(a.workspace);
  const size_t prefix_bytes = align_up((a.num_seqs + 1) * 4, 256);
  const size_t slots = static_cast<size_t>(kMaxDecodeCtas) + a.num_seqs;
  p.ws_prefix = reinterpret_cast<int*>(ws);
  p.ws_ml = reinterpret_cast<float2*>(ws + prefix_bytes);
  p.ws_acc = reinterpret_cast<float*>(ws + prefix_bytes + align_up_sz(slots * a.num_q_heads * 8, 256));
  p.d_status = a.d_status;
  p.L = L;

  auto kern = decode_kernel<T, D, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, L.total, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  // reduce, launched with programmatic stream serialization so its launch
  // overlaps the decode kernel's tail (it waits with griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_seqs);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<T, D>, p, grid);
}

template <typename T>
cudaError_t dispatch_g(const DecodeArgs& a, int group, cudaStream_t stream) {
  const int d = a.pool.head_dim;
#define PA_DEC_CASE(DD, GG) \
  if (d == DD && group == GG) return launch_typed<T, DD, GG>(a, stream);
  PA_DEC_CASE(64, 1) PA_DEC_CASE(64, 2) PA_DEC_CASE(64, 4) PA_DEC_CASE(64, 8)
  PA_DEC_CASE(128, 1) PA_DEC_CASE(128, 2) PA_DEC_CASE(128, 4) PA_DEC_CASE(128, 8)
  PA_DEC_CASE(256, 1) PA_DEC_CASE(256, 2) PA_DEC_CASE(256, 4) PA_DEC_CASE(256, 8)
#undef PA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim) {
  const size_t prefix_bytes = align_up((num_seqs + 1) * 4, 256);
  const size_t slots = static_cast<size_t>(kMaxDecodeCtas) + num_seqs;
  const size_t ml = align_up_sz(slots * num_q_heads * 8, 256);
  const size_t acc = slots * num_q_heads * static_cast<size_t>(head_dim) * 4;
  return prefix_bytes + ml + acc;
}

bool decode_supported(int dtype, int head_dim, int group, int num_kv_heads) {
  if (dtype != PA_F32 && dtype != PA_BF16) return false;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  if (num_kv_heads < 1 || num_kv_heads > kWarps || kWarps % num_kv_heads != 0) return false;
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int group = a.num_q_heads / a.pool.num_kv_heads;
  if (a.pool.dtype == PA_BF16) return dispatch_g<__nv_bfloat16>(a, group, stream);
  return dispatch_g<float>(a, group, stream);
}

}  // namespace pa
