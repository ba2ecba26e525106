// decode_impl.cuh -- paged decode attention on sm_103a (HBM-bound).
// Included by one translation unit per (dtype, head_dim): decode_<dtype>_d<D>.cu.
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
//    into shared memory: 16-byte aligned, fully coalesced (TMA boxes on the
//    tensor-core path below). A 3-4 stage
//    mbarrier pipeline keeps >= 2 blocks (up to 128 KB) in flight per SM. The
//    CTA's slice of the block tables is staged in shared memory up front.
//  * Warps are decoupled: each waits only on the stage it reads, and the last
//    warp to finish a stage (a shared-memory counter) refills it. No CTA-wide
//    barrier runs in the steady state.
//  * bf16 pools with head_dim 64 or 128 and 8 KV heads (one warp each) run
//    both products on the tensor cores with mma.sync m16n8k16 (fp32
//    accumulate): the group's query heads are the rows of a 16-row tile, a
//    block's 16 tokens its columns (Q K^T) and its reduction dimension (P V),
//    the softmax runs on the accumulator fragments and P is re-packed from
//    them as the A operand. A block moves as one 4-D TMA box per 64 columns
//    of head_dim that lands as [head][token][64 elements] with 128-byte
//    swizzle, so the ldmatrix reads of one KV head's tokens hit every bank.
//  * Otherwise (fp32, head_dim 256, fewer KV heads) the products run on the
//    CUDA cores. Warp w serves KV head w % Hkv (and 1/WH of each block's
//    tokens when a KV head has WH > 1 warps). Up to four query heads of the
//    GQA group live in each lane's registers, so one K/V element read from shared memory
//    feeds four FMAs; larger groups split their heads over lane groups.
//    Lanes split a token's head_dim in 16-byte chunks; packed fp32x2 FMAs
//    (FFMA2) do the dot products and the P.V update.
//  * Online softmax in the log2 domain (scores scaled by scale*log2 e) with a
//    lazy running max: the accumulator is rescaled only when a new score
//    exceeds the running max by more than 8 (weights stay <= 256), decided
//    per warp so the rescale is a uniform branch. The partial dot products of
//    a batch are reduce-scattered over the lanes of a token group, so each
//    score's max, weight and sum are computed by one lane only, and the
//    weights are gathered back for P.V.
//  * Two-level cascade (kSib instantiation): a sibling group's members (a
//    request's replies) are walked in entries of up to 16 / G, their query
//    rows packed into the 16-row tile; an entry's shared blocks are read and
//    multiplied once for all of its members, each member's own blocks with
//    the other rows masked. Partials of member m of an entry starting at
//    sequence a, in CTA c of the entry's CTAs c_f .. c_f + n_c - 1, go to slot
//    a + c_f (16 / G) + m n_c + (c - c_f) (c + s without siblings).
//  * Tokens past the context (the tail of a last block) are never loaded by
//    the CUDA-core path; the tensor-core path loads the whole block, masks
//    their scores and zeroes their value rows in shared memory. Either way
//    stale or NaN slots cannot leak into the result.
#pragma once
#include <algorithm>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "tmap.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTableCache = 1024;     // block-table entries staged in shared memory
constexpr float kRescaleThreshold = 8.0f;
// Initial running max of a tensor-core row: finite, so that a row masked for
// a whole block (another member's block) gets weights 2^(-inf - m) = 0, and
// far enough below any score that the first real one replaces it (the
// rescale factor 2^(kNoMax - m) is 0).
constexpr float kNoMax = -1e30f;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 4-D tiled TMA copy global -> shared, completing its bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tmap, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// ldmatrix: four 8 x 8 bf16 matrices; lanes 8i .. 8i+7 give the row
// addresses of matrix i, and lane t receives row t/4, columns 2(t%4), 2(t%4)+1
// of each (the transposed pair with .trans).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// c (16 x 8, fp32) += a (16 x 16, bf16, row-major) * b (16 x 8, bf16, column-major)
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <typename T, int D, int G, int WH>
struct Cfg {
  static constexpr int kHkv = kWarps / WH;
  static constexpr int kElt = sizeof(T);
  static constexpr int kVec = 16 / kElt;             // elements per 16-byte chunk
  static constexpr int kGL = G < 4 ? G : 4;          // query heads per lane
  static constexpr int kHG = G / kGL;                // head groups per token
  static constexpr int kTokPerWarp = kBlockSize / WH;  // tokens of a full block per warp
  // lane slice: q and the accumulator hold kGL * kC floats each (<= 64), and
  // the warp's token slots should not outnumber its tokens per block
  static constexpr int kCq = 64 / kGL;
  static constexpr int kCtok = D * kHG * kTokPerWarp / 32;
  static constexpr int kC0 = kCq < kCtok ? kCq : kCtok;
  static constexpr int kC1 = kC0 < D ? kC0 : D;
  static constexpr int kC = kC1 > kVec ? kC1 : kVec;  // elements per lane per token
  static constexpr int kLpt = D / kC;                 // lanes per (token, head group)
  static constexpr int kLanesTok = kLpt * kHG;        // lanes per token
  static constexpr int kTg = 32 / kLanesTok;          // token slots per warp
  static constexpr int kChunks = kC / kVec;
  static constexpr int kPairs = kC / 2;
  static constexpr int kNt = kTokPerWarp / kTg > 0 ? kTokPerWarp / kTg : 1;
  static constexpr int kBatch = kNt < 4 ? kNt : 4;    // tokens per softmax update per slot
  // Scores of one batch: kN = kBatch x kGL per lane group of kLpt lanes. When
  // they split evenly, a reduce-scatter leaves each lane kR complete scores
  // of one head (kRS); otherwise every lane reduces every score.
  static constexpr int kN = kBatch * kGL;
  static constexpr int kR = kLpt >= 2 && kN % kLpt == 0 ? kN / kLpt : 0;
  static constexpr bool kRS = kR > 0 && kBatch % kR == 0;
  static constexpr int kLh = kRS ? kBatch / kR : 1;  // lanes holding one head's scores
  // the batch's V words are loaded before the score reduction when they fit
  // (at most 8 16-byte words per lane); otherwise just before P.V
  static constexpr bool kPreV = kBatch * kChunks <= 8;
  // bf16 with head_dim 64 or 128 and one warp per KV head runs the products
  // on the tensor cores (mma.sync m16n8k16, fp32 accumulate): the group's
  // query heads are the rows of a 16-row tile, the block's 16 tokens its
  // columns (Q K^T) or its reduction dimension (P V).
  static constexpr bool kMma = sizeof(T) == 2 && (D == 64 || D == 128) && WH == 1 && G <= 16;
  static_assert(kC % kVec == 0, "lane slice must be whole 16-byte chunks");
  static_assert(kLanesTok >= 1 && kLanesTok <= 32 && 32 % kLanesTok == 0, "bad lane split");
  static_assert(G % kGL == 0, "bad head split");
};

struct SmemLayout {
  int stages;
  int tokens_per_unit;  // tokens of one block moved per pipeline stage (16, 8 or 4)
  int parts;            // 16 / tokens_per_unit
  int part_bytes;       // one K (or V) part: tokens_per_unit * Hkv * D * elt
  int off_bars, off_done, off_flags, off_mbars, off_table, off_ntok, off_memb, off_merge, off_prefix,
      off_meta,   // staged cascade metadata (0: not staged)
      off_info;   // per-sequence first block, shared blocks, record (0: not kept)
  int total;
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout make_layout(int stages, int tokens_per_unit, int hkv, int d,
                                                  int elt, int wh, int group, int num_seqs,
                                                  int meta_ints, bool info) {
  SmemLayout L;
  L.stages = stages;
  L.tokens_per_unit = tokens_per_unit;
  L.parts = kBlockSize / tokens_per_unit;
  L.part_bytes = tokens_per_unit * hkv * d * elt;
  const int off = stages * 2 * L.part_bytes;
  L.off_bars = align_up(off, 16);
  L.off_done = L.off_bars + stages * 8;
  L.off_flags = L.off_done + stages * 4;  // [stages] valid tokens, then [stages] member masks
  L.off_mbars = align_up(L.off_flags + stages * 8, 16);   // 2 merge mbarriers per KV head
  L.off_table = align_up(L.off_mbars + 2 * hkv * 8, 16);
  L.off_ntok = L.off_table + kTableCache * 4;  // valid tokens of each cached block
  L.off_memb = L.off_ntok + kTableCache;       // member mask of each cached block (uint16)
  L.off_merge = align_up(L.off_memb + 2 * kTableCache, 16);
  const int merge_bytes = (wh - 1) * hkv * group * (d + 2) * 4;
  L.off_prefix = align_up(L.off_merge + merge_bytes, 16);
  const int end = align_up(L.off_prefix + (num_seqs + 1) * 4, 16);
  L.off_meta = meta_ints > 0 ? end : 0;
  const int end2 = align_up(end + meta_ints * 4, 16);
  L.off_info = info ? end2 : 0;
  L.total = align_up(end2 + (info ? 3 * num_seqs * 4 : 0), 128) + 1024;  // + base alignment
  return L;
}

struct DecodeParams {
  const char* k_pool;
  const char* v_pool;
  int64_t num_blocks;
  int hkv;
  int hq;
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
  // cascade decode (see DecodeArgs); cu_groups == nullptr otherwise
  const int32_t* cu_groups;
  const int32_t* prefix_lens;
  int num_groups;
  const float2* pre_ml;  // [num_seqs, hq]
  const float* pre_acc;  // [num_seqs, hq, D]
  // the prefix partials are computed concurrently (another stream): the
  // decode kernel leaves every cascade sequence as a partial and only the
  // merge kernel, ordered after both, folds the prefix in
  int defer_prefix;
  // nested cascade, second level (tensor-core path only; cu_sib == nullptr
  // otherwise): sequences cu_sib[j] .. cu_sib[j+1]-1 share their first
  // shared_lens[j] tokens (whole blocks, at least the first level's prefix).
  // They are walked in entries of up to sib_m consecutive members whose query
  // rows fill one 16-row MMA tile, so a shared block is read once per entry.
  const int32_t* cu_sib;
  const int32_t* shared_lens;
  int num_sib;
  int sib_m;  // members per entry: 16 / G with sibling groups, else 1
  int64_t num_slots;  // partial slots in the workspace
  // cascade calls: per sequence, written by CTA 0 for the merge kernel: bits
  // 0-3 its offset in its entry, 4-8 the entry's member count, 9 valid
  // lengths, 10 a first-level prefix partial
  uint32_t* ws_rec;
  // tensor-core path: the K and V pools as 4-D maps (see make_tmap_pool_heads)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
};

// The per-sequence inputs the block walk reads (same names as in
// DecodeParams): a cascade call stages them in shared memory, so that the
// prologue's scan and the lookups of every block and entry search on chip.
struct SeqMeta {
  const int32_t* context_lens;
  const int32_t* cu_q_lens;
  const int32_t* cu_groups;
  const int32_t* prefix_lens;
  const int32_t* cu_sib;
  const int32_t* shared_lens;
  int num_seqs, num_rows, max_blocks, num_groups, num_sib, sib_m;
};

// Leading blocks of sequence s whose attention is already in its group's
// shared-prefix partial (0 without groups or outside every group). A prefix
// that is not whole blocks, or longer than the context, is flagged.
template <class P>
__device__ __forceinline__ int prefix_blocks(const P& p, int s, int ctx, bool* bad) {
  if (p.cu_groups == nullptr || p.num_groups <= 0) return 0;
  if (s < p.cu_groups[0] || s >= p.cu_groups[p.num_groups]) return 0;
  const int g = upper_index(p.cu_groups, p.num_groups, s);
  if (s >= p.cu_groups[g + 1]) return 0;
  const int len = p.prefix_lens[g];
  if (len < 0 || len % kBlockSize != 0 || len > ctx) {
    *bad = true;
    return 0;
  }
  return len / kBlockSize;
}

// Sibling group of sequence s (second cascade level), or -1. A group whose
// bounds leave [0, num_seqs] is ignored (its members are walked alone), so
// no entry reaches past the batch.
template <class P>
__device__ __forceinline__ int sib_group(const P& p, int s) {
  if (p.cu_sib == nullptr || p.num_sib <= 0) return -1;
  if (s < p.cu_sib[0] || s >= p.cu_sib[p.num_sib]) return -1;
  const int j = upper_index(p.cu_sib, p.num_sib, s);
  const int g0 = p.cu_sib[j], g1 = p.cu_sib[j + 1];
  return g0 >= 0 && s >= g0 && s < g1 && g1 <= p.num_seqs ? j : -1;
}

// First member of the entry holding sequence s of sibling group j: members
// are taken sib_m at a time from the group's first sequence.
template <class P>
__device__ __forceinline__ int entry_start(const P& p, int j, int s) {
  const int g0 = p.cu_sib[j];
  return g0 + (s - g0) / p.sib_m * p.sib_m;
}

// The CTA whose range holds block b of the decode order (B blocks, `grid`
// CTAs; CTA c holds blocks [c B / grid, (c + 1) B / grid)).
__host__ __device__ __forceinline__ int64_t cta_of_block(int64_t b, int64_t B, int64_t grid) {
  return ((b + 1) * grid - 1) / B;
}

// What the block walk needs to know about sequence s, worked out in one pass:
// the blocks the decode kernel reads for it (0 when s is not a decode
// sequence or its lengths are invalid), where they start in its block table,
// and its sibling entry. A sibling group's shared blocks after the
// first-level prefix are counted once per entry, as the first blocks of its
// first member (every member's rows attend them); the other members count
// only their own blocks.
struct SeqInfo {
  int blocks;   // blocks read for s
  int first;    // logical block of s's table where they start
  int nsh;      // how many of them are the entry's shared blocks
  int off, k;   // s is member `off` of an entry of k members
  bool bad;     // invalid lengths (the row is zeroed and flagged)
  bool has_pre; // the attention over a first-level prefix is a separate partial
};
template <class P>
__device__ __forceinline__ SeqInfo seq_info(const P& p, int s) {
  SeqInfo r;
  r.blocks = 0;
  r.first = 0;
  r.nsh = 0;
  r.off = 0;
  r.k = 1;
  r.bad = false;
  r.has_pre = false;
  int q_len = 1;
  if (p.cu_q_lens != nullptr) {
    q_len = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
    if (q_len < 0 || p.cu_q_lens[s] < 0 || p.cu_q_lens[s + 1] > p.num_rows) {
      r.bad = true;  // malformed cu_q_lens: never index q/out with it
      return r;
    }
  }
  if (q_len != 1) return r;
  const int ctx = p.context_lens[s];
  if (ctx < 1 || ctx > p.max_blocks * kBlockSize) {
    r.bad = true;
    return r;
  }
  bool bad_prefix = false;
  const int skip = prefix_blocks(p, s, ctx, &bad_prefix);
  if (bad_prefix) {
    r.bad = true;
    return r;
  }
  r.first = skip;
  r.has_pre = skip > 0;
  const int j = sib_group(p, s);
  if (j < 0) {
    r.blocks = (ctx + kBlockSize - 1) / kBlockSize - skip;
    return r;
  }
  const int a = entry_start(p, j, s);
  r.off = s - a;
  r.k = min(p.sib_m, p.cu_sib[j + 1] - a);
  // the shared blocks are read through the entry's first member's table: its
  // lengths must hold them too, with the same first-level prefix
  const int shared = p.shared_lens[j];
  if (shared < skip * kBlockSize || shared % kBlockSize != 0 || shared > ctx) {
    r.bad = true;
    return r;
  }
  if (a != s) {
    const int ctx_a = p.context_lens[a];
    bool bad_a = false;
    if (ctx_a < 1 || ctx_a > p.max_blocks * kBlockSize || shared > ctx_a ||
        prefix_blocks(p, a, ctx_a, &bad_a) != skip || bad_a) {
      r.bad = true;
      return r;
    }
  }
  const int se = shared / kBlockSize;
  r.nsh = a == s ? se - skip : 0;
  if (a != s) r.first = se;
  r.blocks = (ctx + kBlockSize - 1) / kBlockSize - se + r.nsh;
  return r;
}

// SeqInfo packed for the merge kernel and the shared-memory table: bits 0-3
// the member offset, 4-8 the entry size, 9 valid lengths, 10 a first-level
// prefix partial.
__device__ __forceinline__ uint32_t pack_rec(const SeqInfo& r) {
  return static_cast<uint32_t>(r.off) | (static_cast<uint32_t>(r.k) << 4) | (r.bad ? 0u : 1u << 9) |
         (r.has_pre ? 1u << 10 : 0u);
}
__device__ __forceinline__ int rec_off(uint32_t rec) { return static_cast<int>(rec & 15u); }
__device__ __forceinline__ int rec_k(uint32_t rec) { return static_cast<int>((rec >> 4) & 31u); }
__device__ __forceinline__ bool rec_valid(uint32_t rec) { return (rec >> 9) & 1u; }
__device__ __forceinline__ bool rec_pre(uint32_t rec) { return (rec >> 10) & 1u; }

// Blocks the decode kernel reads for sequence s; sets *bad for invalid lengths.
template <class P>
__device__ __forceinline__ int decode_blocks(const P& p, int s, bool* bad) {
  const SeqInfo r = seq_info(p, s);
  if (r.bad) *bad = true;
  return r.blocks;
}

__device__ __forceinline__ int query_row(const DecodeParams& p, int s) {
  return p.cu_q_lens != nullptr ? p.cu_q_lens[s] : s;
}

// 16 bytes of T as fp32 pairs.
template <typename T>
__device__ __forceinline__ void unpack_pairs(const uint4 raw, float2* dst) {
  if constexpr (sizeof(T) == 2) {
    dst[0] = bf16x2_to_float2(raw.x);
    dst[1] = bf16x2_to_float2(raw.y);
    dst[2] = bf16x2_to_float2(raw.z);
    dst[3] = bf16x2_to_float2(raw.w);
  } else {
    dst[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
    dst[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
  }
}

// 16 bytes of T from shared memory as fp32 pairs.
template <typename T>
__device__ __forceinline__ void load_pairs(const T* src, float2* dst) {
  unpack_pairs<T>(*reinterpret_cast<const uint4*>(src), dst);
}

// Rescale factor of a partial with running max m when the merged max is mn.
__device__ __forceinline__ float merge_factor(float m, float mn) {
  return m == -INFINITY ? 0.f : fast_exp2(m - mn);
}

// kSib: the nested cascade's sibling entries (tensor-core path only); the
// other instantiation walks one sequence per entry with none of their
// bookkeeping (row masks, member records, entry slots) in its loops.
template <typename T, int D, int G, int WH, bool kSib>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = Cfg<T, D, G, WH>;
  static_assert(!kSib || C::kMma, "sibling entries run on the tensor-core path");
  constexpr int HKV = C::kHkv;
  extern __shared__ __align__(128) char smem_raw[];
  // 1024-byte aligned base (128-byte swizzled TMA boxes need it)
  char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const SmemLayout& L = p.L;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.off_bars);
  int* done = reinterpret_cast<int*>(smem + L.off_done);
  int* flags = reinterpret_cast<int*>(smem + L.off_flags);
  uint32_t* memb = reinterpret_cast<uint32_t*>(flags + L.stages);  // rows of the entry per stage
  uint64_t* merge_full = reinterpret_cast<uint64_t*>(smem + L.off_mbars);
  uint64_t* merge_empty = merge_full + HKV;
  int* table = reinterpret_cast<int*>(smem + L.off_table);
  uint8_t* block_ntok = reinterpret_cast<uint8_t*>(smem + L.off_ntok);
  uint16_t* block_memb = reinterpret_cast<uint16_t*>(smem + L.off_memb);
  float* merge = reinterpret_cast<float*>(smem + L.off_merge);
  int* prefix = reinterpret_cast<int*>(smem + L.off_prefix);
  __shared__ int warp_sums[kWarps];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int S = p.num_seqs;

  if (tid == 0) {
    for (int i = 0; i < L.stages; ++i) {
      mbar_init(&bars[i], 1);
      done[i] = 0;
    }
    for (int i = 0; i < HKV; ++i) {
      mbar_init(&merge_full[i], WH - 1 > 0 ? WH - 1 : 1);
      mbar_init(&merge_empty[i], 1);
    }
    fence_mbar_init();
  }
  // the block walk's per-sequence inputs: staged in shared memory for a
  // cascade call (context lengths, group and sibling bounds and lengths)
  __shared__ SeqMeta meta;
  if (L.off_meta > 0) {
    int32_t* m_ctx = reinterpret_cast<int32_t*>(smem + L.off_meta);
    int32_t* m_cu = m_ctx + S;
    int32_t* m_pl = m_cu + (p.num_groups > 0 ? p.num_groups + 1 : 0);
    int32_t* m_sib = m_pl + (p.num_groups > 0 ? p.num_groups : 0);
    int32_t* m_sl = m_sib + (p.num_sib > 0 ? p.num_sib + 1 : 0);
    // the five arrays lie back to back from m_ctx: one index space, eight
    // loads in flight per thread before their stores (loads issued one by
    // one would each wait out a round trip to a busy HBM)
    const int n0 = S, n1 = static_cast<int>(m_pl - m_ctx), n2 = static_cast<int>(m_sib - m_ctx),
              n3 = static_cast<int>(m_sl - m_ctx), n4 = n3 + (p.num_sib > 0 ? p.num_sib : 0);
    auto src_at = [&](int i) -> int32_t {
      if (i < n0) return __ldg(p.context_lens + i);
      if (i < n1) return __ldg(p.cu_groups + (i - n0));
      if (i < n2) return __ldg(p.prefix_lens + (i - n1));
      if (i < n3) return __ldg(p.cu_sib + (i - n2));
      return __ldg(p.shared_lens + (i - n3));
    };
    constexpr int kBatch = 8;
    for (int base = 0; base < n4; base += kBatch * kThreads) {
      int32_t v[kBatch];
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int i = base + r * kThreads + tid;
        v[r] = i < n4 ? src_at(i) : 0;
      }
#pragma unroll
      for (int r = 0; r < kBatch; ++r) {
        const int i = base + r * kThreads + tid;
        if (i < n4) m_ctx[i] = v[r];
      }
    }
    if (tid == 0) {
      meta.context_lens = m_ctx;
      meta.cu_groups = p.num_groups > 0 ? m_cu : p.cu_groups;
      meta.prefix_lens = p.num_groups > 0 ? m_pl : p.prefix_lens;
      meta.cu_sib = p.num_sib > 0 ? m_sib : p.cu_sib;
      meta.shared_lens = p.num_sib > 0 ? m_sl : p.shared_lens;
    }
  } else if (tid == 0) {
    meta.context_lens = p.context_lens;
    meta.cu_groups = p.cu_groups;
    meta.prefix_lens = p.prefix_lens;
    meta.cu_sib = p.cu_sib;
    meta.shared_lens = p.shared_lens;
  }
  if (tid == 0) {
    meta.cu_q_lens = p.cu_q_lens;
    meta.num_seqs = S;
    meta.num_rows = p.num_rows;
    meta.max_blocks = p.max_blocks;
    meta.num_groups = p.num_groups;
    meta.num_sib = p.num_sib;
    meta.sib_m = p.sib_m;
  }
  __syncthreads();
  // Each sequence's SeqInfo, worked out once per CTA: kept in shared memory
  // when it fits (then the block counts are scanned in place), else worked
  // out again wherever it is needed.
  int* s_first = L.off_info > 0 ? reinterpret_cast<int*>(smem + L.off_info) : nullptr;
  int* s_nsh = L.off_info > 0 ? s_first + S : nullptr;
  uint32_t* s_rec = L.off_info > 0 ? reinterpret_cast<uint32_t*>(s_nsh + S) : nullptr;
  bool bad_len = false;
  if (s_first != nullptr) {
    const SeqMeta m = meta;  // in registers for the scan
    for (int s = tid; s < S; s += kThreads) {
      const SeqInfo r = seq_info(m, s);
      prefix[s] = r.blocks;
      s_first[s] = r.first;
      s_nsh[s] = r.nsh;
      s_rec[s] = pack_rec(r);
      bad_len |= r.bad;
    }
    __syncthreads();
    block_exclusive_scan<kThreads>(S, [&](int s) { return prefix[s]; }, prefix, warp_sums);
  } else {
    block_exclusive_scan<kThreads>(
        S, [&](int s) { return decode_blocks(meta, s, &bad_len); }, prefix, warp_sums);
  }
  if (bad_len && blockIdx.x == 0) status_or(p.d_status, PA_STATUS_BAD_LENGTH);
  // the record of a sequence that has blocks to read: without groups or
  // sibling groups it is the same for all (member 0 of a one-member entry,
  // valid, no prefix partial), else kept or worked out again
  const bool plain = p.cu_groups == nullptr && p.cu_sib == nullptr;
  auto rec_of = [&](int s) -> uint32_t {
    if (s_first != nullptr) return s_rec[s];
    if (plain) return (1u << 4) | (1u << 9);
    return pack_rec(seq_info(meta, s));
  };
  // logical block j of sequence s, and the rows of its entry that attend it,
  // for block b of the decode order
  auto locate = [&](int64_t b, int* s_out, int* j_out, uint32_t* rows_out) {
    const int s = upper_index(prefix, S, b);
    const int r = static_cast<int>(b - prefix[s]);
    int first, nsh;
    uint32_t rec;
    if (s_first != nullptr) {
      first = s_first[s];
      nsh = s_nsh[s];
      rec = s_rec[s];
    } else if (plain) {  // the table lookup need not wait for the lengths
      first = 0;
      nsh = 0;
      rec = rec_of(s);
    } else {
      const SeqInfo si = seq_info(meta, s);
      first = si.first;
      nsh = si.nsh;
      rec = pack_rec(si);
    }
    *s_out = s;
    *j_out = first + r;
    *rows_out = r < nsh ? (1u << rec_k(rec)) - 1u : 1u << rec_off(rec);
  };

  // cascade calls: the merge kernel's per-sequence record (see DecodeParams)
  if (blockIdx.x == 0 && p.ws_rec != nullptr)
    for (int s = tid; s < S; s += kThreads)
      p.ws_rec[s] = s_first != nullptr ? s_rec[s] : pack_rec(seq_info(meta, s));

  // Invalid decode sequences (bad lengths) get zero output rows, written once:
  // one warp of the grid checks each sequence, so no CTA lags the others
  for (int s = blockIdx.x * kWarps + warp; s < S; s += gridDim.x * kWarps) {
    const bool bad = s_first != nullptr ? !rec_valid(s_rec[s]) : seq_info(meta, s).bad;
    int q_len = 1;
    if (p.cu_q_lens != nullptr) q_len = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
    const int row = query_row(p, s);
    if (bad && q_len == 1 && row >= 0 && row < p.num_rows) {
      T* o = static_cast<T*>(p.out) + static_cast<int64_t>(row) * p.hq * D;
      for (int i = lane; i < p.hq * D; i += 32) o[i] = from_float<T>(0.f);
    }
  }
  if (blockIdx.x == 0)
    for (int i = tid; i <= S; i += kThreads) p.ws_prefix[i] = prefix[i];

  const int64_t B = prefix[S];
  const int64_t grid = gridDim.x;
  const int64_t lo = static_cast<int64_t>(blockIdx.x) * B / grid;
  const int64_t hi = (static_cast<int64_t>(blockIdx.x) + 1) * B / grid;
  if (lo >= hi) return;

  const int parts = L.parts;
  const int tpu = L.tokens_per_unit;
  const int64_t n_units = (hi - lo) * parts;
  constexpr int kTokenBytes = HKV * D * C::kElt;

  // Issue unit u into stage st (= u % stages; the caller keeps it), called
  // by one lane; `direct` reads the block table in global memory instead of
  // the staged slice.
  auto issue = [&](int u, int st, bool direct) {
    const int rel = parts == 1 ? u : u / parts;  // block of the CTA's range
    const int part = parts == 1 ? 0 : u % parts;
    int phys, block_tokens;
    uint32_t rows;
    if (rel < kTableCache && !direct) {
      phys = table[rel];
      block_tokens = block_ntok[rel];
      rows = kSib ? block_memb[rel] : 1u;
    } else {
      int s, j;
      locate(lo + rel, &s, &j, &rows);
      phys = p.block_tables[static_cast<int64_t>(s) * p.max_blocks + j];
      block_tokens = min(kBlockSize, meta.context_lens[s] - j * kBlockSize);
      if (direct && rel < kTableCache) {  // staged here, not again below
        table[rel] = phys;
        block_ntok[rel] = static_cast<uint8_t>(block_tokens);
        if constexpr (kSib) block_memb[rel] = static_cast<uint16_t>(rows);
      }
    }
    if constexpr (kSib) memb[st] = rows;
    const int ntok = min(tpu, block_tokens - part * tpu);
    if (phys < 0 || phys >= p.num_blocks) {
      flags[st] = -1;
      status_or(p.d_status, PA_STATUS_BAD_BLOCK);
      mbar_arrive(&bars[st]);
    } else if (ntok <= 0) {
      flags[st] = 0;
      mbar_arrive(&bars[st]);
    } else {
      flags[st] = ntok;
      const uint32_t bytes = static_cast<uint32_t>(ntok * kTokenBytes);
      const int64_t src = (static_cast<int64_t>(phys) * kBlockSize + part * tpu) * kTokenBytes;
      char* kdst = smem + st * 2 * L.part_bytes;
      if constexpr (C::kMma) {
        // the whole block, one 16 KB box per 64 columns of head_dim: [head][token][64]
        // with 128-byte swizzle; slots past the context come along and are masked
        constexpr uint32_t kBox = 64 * kBlockSize * HKV * 2;
        mbar_arrive_expect_tx(&bars[st], 2 * (D / 64) * kBox);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_4d(kdst + h * kBox, &p.tm_k, 64 * h, 0, 0, phys, &bars[st]);
          tma_load_4d(kdst + L.part_bytes + h * kBox, &p.tm_v, 64 * h, 0, 0, phys, &bars[st]);
        }
      } else {
        mbar_arrive_expect_tx(&bars[st], 2 * bytes);
        bulk_g2s(kdst, p.k_pool + src, bytes, &bars[st]);
        bulk_g2s(kdst + L.part_bytes, p.v_pool + src, bytes, &bars[st]);
      }
    }
  };
  // the first stages are issued from the global table at once, so their
  // copies are in flight while the CTA stages the rest of its table slice;
  // one thread each, so their table lookups overlap
  const int n_first = static_cast<int>(min(static_cast<int64_t>(L.stages), n_units));
  if (tid < n_first) issue(tid, tid, true);

  // stage this CTA's slice of the block tables (first kTableCache blocks)
  // with the number of context tokens each block holds (the first n_first
  // blocks were staged by their issue above; with parts > 1 a unit is a part
  // of a block, and unit tid's block is tid / parts)
  const int n_cached = static_cast<int>(min(hi - lo, static_cast<int64_t>(kTableCache)));
  for (int i = tid + (parts == 1 && tid < n_first ? kThreads : 0); i < n_cached; i += kThreads) {
    int s, j;
    uint32_t rows;
    locate(lo + i, &s, &j, &rows);
    table[i] = p.block_tables[static_cast<int64_t>(s) * p.max_blocks + j];
    block_ntok[i] = static_cast<uint8_t>(min(kBlockSize, meta.context_lens[s] - j * kBlockSize));
    if constexpr (kSib) block_memb[i] = static_cast<uint16_t>(rows);
  }
  __syncthreads();
  // the merge kernel may be launched now: it waits (griddepcontrol.wait) for
  // this whole grid to complete before it reads anything
  pdl_launch_dependents();

  if constexpr (C::kMma) {
    // -------------------------------------------------- tensor-core consumers
    // Warp g serves KV head g. Per block: S (16 rows x 16 tokens) = Q K^T in
    // D / 16 k-steps, each two m16n8k16 MMAs; the online softmax runs on the
    // S fragments in fp32; O (16 rows x D) += P V with P re-packed from the S
    // fragments as the A operand. Rows are the group's query heads (G of 16
    // are real), so lane t owns rows t/4 and t/4 + 8, columns 2(t%4), +1.
    // A block arrives as one TMA box per 64 columns of head_dim, laid out
    // [head][token][64 elements] with 128-byte swizzle (the 16-byte chunk
    // index XOR the token's row within its 8-row atom), so the 8 tokens of
    // one ldmatrix matrix hit 8 different bank groups.
    const int g = warp;
    const int gi = lane >> 2, qi = lane & 3;
    constexpr int KS = D / 16;
    constexpr uint32_t kBox = 64 * kBlockSize * HKV * 2;
    // ldmatrix rows of this lane: K matrices are (tokens 0-7 | 8-15) x
    // (d lo | hi) of a k-step, V (.trans) matrices are (tokens 0-7 | 8-15) x
    // (d of n-tile 2n | 2n+1); column n of S n-tile j is token 8j + n
    const int lm = lane >> 3, lr = lane & 7;
    const int tk = (lm >> 1) * 8 + lr, tv = (lm & 1) * 8 + lr;
    const uint32_t k_row = static_cast<uint32_t>((g * kBlockSize + tk) * 128);
    const uint32_t v_row = static_cast<uint32_t>((g * kBlockSize + tv) * 128);
    const uint32_t sbase = smem_addr(smem);
    uint32_t qa[KS][4];
    float o[D / 8][4];
    int u = 0;
    int st_c = 0;
    uint32_t ph_c = 0;
    // tile rows gi and gi + 8 of this lane: query head (row % G) of member
    // (row / G) of the current entry
    const int mr0 = gi / G, mr1 = (gi + 8) / G;
    int s = upper_index(prefix, S, lo);
    bool ok = true;
    while (u < n_units && ok) {
      while (prefix[s + 1] <= lo + (parts == 1 ? u : u / parts)) ++s;
      // the entry holding s: members a .. a + k - 1, blocks [e_lo, e_hi)
      const uint32_t rec_s = rec_of(s);
      const int a = kSib ? s - rec_off(rec_s) : s, k = kSib ? rec_k(rec_s) : 1;
      const int64_t e_lo = prefix[a], e_hi = prefix[a + k];
      // units from here to the end of the entry or of the range (counted from
      // the current unit, so that even inconsistent sibling bounds cannot
      // make the walk repeat or overrun units)
      const int64_t seq_units = (min(hi, e_hi) - lo) * parts - u;
      const bool whole = e_lo >= lo && e_hi <= hi;
      // members with valid lengths (a member with bad ones may sit in an
      // entry whose shared blocks are read; its row stays zero) and members
      // with a first-level prefix partial, one lane per member
      uint32_t vmask = 1u, pmask = rec_pre(rec_s) ? 1u : 0u;
      if constexpr (kSib) {
        bool v = false, hp = false;
        if (lane < k) {
          const uint32_t rm = rec_of(a + lane);
          v = rec_valid(rm);
          hp = rec_pre(rm);
        }
        vmask = __ballot_sync(0xffffffffu, v);
        pmask = __ballot_sync(0xffffffffu, hp);
      }
      // Q as stored (bf16 pairs); the scale is applied to the fp32 scores
      if constexpr (!kSib) {
        const uint32_t* q = reinterpret_cast<const uint32_t*>(static_cast<const T*>(p.q) +
                                                              static_cast<int64_t>(query_row(p, s)) * p.hq * D);
        const int h0 = g * G + gi, h1 = g * G + gi + 8;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int c = (16 * kk + 2 * qi) / 2;  // bf16-pair index
          qa[kk][0] = gi < G ? __ldg(q + h0 * (D / 2) + c) : 0u;
          qa[kk][1] = gi + 8 < G ? __ldg(q + h1 * (D / 2) + c) : 0u;
          qa[kk][2] = gi < G ? __ldg(q + h0 * (D / 2) + c + 4) : 0u;
          qa[kk][3] = gi + 8 < G ? __ldg(q + h1 * (D / 2) + c + 4) : 0u;
        }
      } else {
        const bool in0 = mr0 < k, in1 = mr1 < k;
        const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
            static_cast<const T*>(p.q) + static_cast<int64_t>(query_row(p, a + (in0 ? mr0 : 0))) * p.hq * D);
        const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
            static_cast<const T*>(p.q) + static_cast<int64_t>(query_row(p, a + (in1 ? mr1 : 0))) * p.hq * D);
        const int h0 = g * G + gi % G, h1 = g * G + (gi + 8) % G;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int c = (16 * kk + 2 * qi) / 2;  // bf16-pair index
          qa[kk][0] = in0 ? __ldg(q0 + h0 * (D / 2) + c) : 0u;
          qa[kk][1] = in1 ? __ldg(q1 + h1 * (D / 2) + c) : 0u;
          qa[kk][2] = in0 ? __ldg(q0 + h0 * (D / 2) + c + 4) : 0u;
          qa[kk][3] = in1 ? __ldg(q1 + h1 * (D / 2) + c + 4) : 0u;
        }
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      // a sibling entry's rows start from a finite running max (kNoMax)
      float m0 = kSib ? kNoMax : -INFINITY, m1 = kSib ? kNoMax : -INFINITY, l0 = 0.f, l1 = 0.f;
      uint32_t poison = 0;  // members whose rows met a bad block

      for (int su = 0; su < seq_units; ++su, ++u) {
        const int st = st_c;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], ph_c));
        if (!ok) break;
        const int ntok = flags[st];
        if (ntok < 0) poison |= kSib ? memb[st] : 1u;
        if (ntok > 0) {
          const uint32_t kb = sbase + static_cast<uint32_t>(st * 2 * L.part_bytes);
          const uint32_t vb = kb + static_cast<uint32_t>(L.part_bytes);
          if (ntok < kBlockSize) {
            // slots past the context hold stale or poisoned values: zero this
            // head's value rows there (their weight is 0, and 0 x NaN is NaN)
            char* vpart = smem + st * 2 * L.part_bytes + L.part_bytes;
            constexpr int kChunkRow = D * 2 / 16;  // 16-byte chunks of one row over all boxes
            for (int i = lane; i < (kBlockSize - ntok) * kChunkRow; i += 32) {
              const int t = ntok + i / kChunkRow, c = i % kChunkRow;
              *reinterpret_cast<uint4*>(vpart + (c / 8) * kBox + (g * kBlockSize + t) * 128 + (c % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // ordered before the stage's next TMA copy
            __syncwarp();
          }
          float sc[2][4];
#pragma unroll
          for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            uint32_t kf[4];
            const uint32_t c = static_cast<uint32_t>(2 * (kk & 3) + (lm & 1));
            ldsm_x4(kb + (kk >> 2) * kBox + k_row + ((c ^ (tk & 7)) << 4), kf);
            mma_16816(sc[0], qa[kk], kf[0], kf[1]);
            mma_16816(sc[1], qa[kk], kf[2], kf[3]);
          }
          // log2-domain scores; tokens past the context, and every token for
          // rows of members that do not attend this block (another member's
          // own block), are masked
          int nt0 = ntok, nt1 = ntok;
          if constexpr (kSib) {
            const uint32_t rows = memb[st];
            nt0 = (rows >> mr0) & 1u ? ntok : 0;
            nt1 = (rows >> mr1) & 1u ? ntok : 0;
          }
          float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = 8 * n + 2 * qi + e;  // token of column 2qi+e of n-tile n
              sc[n][e] = col < nt0 ? sc[n][e] * p.scale_log2 : -INFINITY;
              sc[n][2 + e] = col < nt1 ? sc[n][2 + e] * p.scale_log2 : -INFINITY;
              mt0 = fmaxf(mt0, sc[n][e]);
              mt1 = fmaxf(mt1, sc[n][2 + e]);
            }
#pragma unroll
          for (int off = 1; off <= 2; off <<= 1) {
            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
          }
          // lazy running max: moved only when a score exceeds it by more than 8
          const bool need0 = mt0 > m0 + kRescaleThreshold, need1 = mt1 > m1 + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need0 || need1)) {
            const float n0 = need0 ? mt0 : m0, n1 = need1 ? mt1 : m1;
            // 0 from -inf (plain) or kNoMax (sibling entries)
            const float a0 = (!kSib && m0 == -INFINITY) ? 0.f : fast_exp2(m0 - n0);
            const float a1 = (!kSib && m1 == -INFINITY) ? 0.f : fast_exp2(m1 - n1);
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              o[n][0] *= a0;
              o[n][1] *= a0;
              o[n][2] *= a1;
              o[n][3] *= a1;
            }
            m0 = n0;
            m1 = n1;
          }
          float w[2][4];
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            w[n][0] = fast_exp2(sc[n][0] - m0);
            w[n][1] = fast_exp2(sc[n][1] - m0);
            w[n][2] = fast_exp2(sc[n][2] - m1);
            w[n][3] = fast_exp2(sc[n][3] - m1);
          }
          l0 += (w[0][0] + w[0][1]) + (w[1][0] + w[1][1]);
          l1 += (w[0][2] + w[0][3]) + (w[1][2] + w[1][3]);
          const uint32_t pa[4] = {pack_bf16x2(w[0][0], w[0][1]), pack_bf16x2(w[0][2], w[0][3]),
                                  pack_bf16x2(w[1][0], w[1][1]), pack_bf16x2(w[1][2], w[1][3])};
#pragma unroll
          for (int np = 0; np < KS; ++np) {
            uint32_t vf[4];
            const uint32_t c = static_cast<uint32_t>(2 * (np & 3) + (lm >> 1));
            ldsm_x4_trans(vb + (np >> 2) * kBox + v_row + ((c ^ (tv & 7)) << 4), vf);
            mma_16816(o[2 * np], pa, vf[0], vf[1]);
            mma_16816(o[2 * np + 1], pa, vf[2], vf[3]);
          }
        }
        // stage consumed by this warp; the last warp to finish refills it
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          const int prev = atomicAdd(&done[st], 1);
          if (prev == kWarps - 1) {
            done[st] = 0;
            __threadfence_block();
            if (u + L.stages < n_units) issue(u + L.stages, st, false);
          }
        }
        if (++st_c == L.stages) {
          st_c = 0;
          ph_c ^= 1;
        }
      }
      if (!ok) break;

      // ------------------------------------------------------------ finish s
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      // partial slots of the entry: member m in CTA c (c_f <= c < c_f + n_c)
      // writes slot a + c_f sib_m + m n_c + (c - c_f), unique over the batch
      // since entries and CTA ranges are both in block order (c + s without
      // sibling groups)
      int64_t slot_c = static_cast<int64_t>(blockIdx.x) + s, n_c = 0;  // member 0's slot
      if constexpr (kSib) {
        const int64_t c_f = cta_of_block(e_lo, prefix[S], gridDim.x);
        n_c = cta_of_block(e_hi - 1, prefix[S], gridDim.x) - c_f + 1;
        slot_c = a + c_f * p.sib_m + (static_cast<int64_t>(blockIdx.x) - c_f);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int mr = r ? mr1 : mr0;  // member of the entry
        if (mr >= k || !((vmask >> mr) & 1u)) continue;
        const int sq = a + mr;
        const int row = query_row(p, sq);
        const bool has_pre = (pmask >> mr) & 1u;
        const bool poisoned = (poison >> mr) & 1u;
        const int head = g * G + (gi + 8 * r) % G;
        const float mx = r ? m1 : m0;
        float lr_ = r ? l1 : l0;
        if (whole && !(has_pre && p.defer_prefix)) {
          bool pre_poisoned = false;
          if (has_pre) {
            // fold in the shared-prefix partial of this sequence
            const int64_t idx = static_cast<int64_t>(sq) * p.hq + head;
            const float2 pml = p.pre_ml[idx];
            pre_poisoned = pml.y < 0.f;
            const float mn = fmaxf(mx, pml.x);
            const float fa = merge_factor(mx, mn), fb = merge_factor(pml.x, mn);
            lr_ = lr_ * fa + pml.y * fb;
            const float* prow = p.pre_acc + idx * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              const float2 pv = *reinterpret_cast<const float2*>(prow + 8 * n + 2 * qi);
              o[n][2 * r] = o[n][2 * r] * fa + pv.x * fb;
              o[n][2 * r + 1] = o[n][2 * r + 1] * fa + pv.y * fb;
            }
          }
          const float inv = (poisoned || pre_poisoned) ? 0.f : 1.f / lr_;
          uint32_t* orow = reinterpret_cast<uint32_t*>(static_cast<T*>(p.out) +
                                                       (static_cast<int64_t>(row) * p.hq + head) * D);
#pragma unroll
          for (int n = 0; n < D / 8; ++n)
            orow[4 * n + qi] = pack_bf16x2(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
        } else {
          const int64_t slot = slot_c + mr * n_c;
          if (slot < 0 || slot >= p.num_slots) continue;  // only with inconsistent sibling bounds
          if (qi == 0) p.ws_ml[slot * p.hq + head] = make_float2(mx, poisoned ? -1.f : lr_);
          float* arow = p.ws_acc + (slot * p.hq + head) * D;
#pragma unroll
          for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<float2*>(arow + 8 * n + 2 * qi) = make_float2(o[n][2 * r], o[n][2 * r + 1]);
        }
      }
    }
    if (!ok && lane == 0) status_or(p.d_status, PA_STATUS_TIMEOUT);
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int g = warp % HKV;     // this warp's KV head
  const int sub = warp / HKV;   // which share of a block's tokens
  const int tg = lane / C::kLanesTok;                  // token slot
  const int hg = (lane / C::kLpt) % C::kHG;            // head group
  const int kl = lane % C::kLpt;                       // chunk column
  const int head0 = g * G + hg * C::kGL;               // first query head of this lane

  float2 qf[C::kGL][C::kPairs];
  float2 acc[C::kGL][C::kPairs];
  float m[C::kGL], l[C::kGL];
  float l_own = 0.f;            // reduce-scatter: the sum of this lane's own head
  const int base = lane - kl;   // first lane of this (token slot, head group)
  const int own_j = kl * (C::kRS ? C::kR : 0);  // first score this lane owns
  const int own_h = C::kRS ? own_j / C::kBatch : 0;
  const int own_b = C::kRS ? own_j % C::kBatch : 0;
  int merges = 0;  // sequences merged across warps so far (mbarrier phase)

  int u = 0;
  int st_c = 0;       // stage of unit u (u % stages) and its mbarrier phase,
  uint32_t ph_c = 0;  // kept incrementally: no division per unit
  int s = upper_index(prefix, S, lo);
  bool ok = true;
  while (u < n_units && ok) {
    while (prefix[s + 1] <= lo + (parts == 1 ? u : u / parts)) ++s;
    const int64_t seq_lo = max(lo, static_cast<int64_t>(prefix[s]));
    const int64_t seq_hi = min(hi, static_cast<int64_t>(prefix[s + 1]));
    const int64_t seq_units = (seq_hi - seq_lo) * parts;
    const bool whole = prefix[s] >= lo && prefix[s + 1] <= hi;
    const int row = query_row(p, s);
    const bool has_pre = rec_pre(rec_of(s));

    // this lane's query heads, pre-scaled into the log2 domain
    {
      const T* qrow = static_cast<const T*>(p.q) + (static_cast<int64_t>(row) * p.hq + head0) * D;
#pragma unroll
      for (int h = 0; h < C::kGL; ++h) {
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          float2 pr[C::kVec / 2];
          const uint4 raw =
              __ldg(reinterpret_cast<const uint4*>(qrow + h * D + (kl + C::kLpt * c) * C::kVec));
          if constexpr (sizeof(T) == 2) {
            pr[0] = bf16x2_to_float2(raw.x);
            pr[1] = bf16x2_to_float2(raw.y);
            pr[2] = bf16x2_to_float2(raw.z);
            pr[3] = bf16x2_to_float2(raw.w);
          } else {
            pr[0] = make_float2(__uint_as_float(raw.x), __uint_as_float(raw.y));
            pr[1] = make_float2(__uint_as_float(raw.z), __uint_as_float(raw.w));
          }
#pragma unroll
          for (int i = 0; i < C::kVec / 2; ++i)
            qf[h][c * (C::kVec / 2) + i] = make_float2(pr[i].x * p.scale_log2, pr[i].y * p.scale_log2);
        }
        m[h] = -INFINITY;
        l[h] = 0.f;
        l_own = 0.f;
#pragma unroll
        for (int i = 0; i < C::kPairs; ++i) acc[h][i] = make_float2(0.f, 0.f);
      }
    }
    bool poisoned = false;

    for (int su = 0; su < seq_units; ++su, ++u) {
      const int st = st_c;
      const uint32_t parity = ph_c;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], parity));
      if (!ok) break;
      const int ntok = flags[st];
      if (ntok < 0) poisoned = true;
      const T* kbase = reinterpret_cast<const T*>(smem + st * 2 * L.part_bytes);
      const T* vbase = reinterpret_cast<const T*>(smem + st * 2 * L.part_bytes + L.part_bytes);
      // token of slot tg at step i: sub + WH * (tg + kTg * i)
      for (int i0 = 0; sub + WH * (C::kTg * i0) < ntok; i0 += C::kBatch) {
        float sc[C::kBatch][C::kGL];
        const bool full = sub + WH * (C::kTg - 1 + C::kTg * (i0 + C::kBatch - 1)) < ntok;
#pragma unroll
        for (int b = 0; b < C::kBatch; ++b) {
          const int t = sub + WH * (tg + C::kTg * (i0 + b));
          float2 part[C::kGL];
#pragma unroll
          for (int h = 0; h < C::kGL; ++h) part[h] = make_float2(0.f, 0.f);
          {
            // loaded whether or not the token is valid (the score of a token
            // past ntok is never used), so the loads need not wait for ntok;
            // the row index stays inside the unit
            const int tl = t < tpu ? t : tpu - 1;
            const T* krow = kbase + (tl * HKV + g) * D;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              float2 kf[C::kVec / 2];
              load_pairs(krow + (kl + C::kLpt * c) * C::kVec, kf);
#pragma unroll
              for (int i = 0; i < C::kVec / 2; ++i)
#pragma unroll
                for (int h = 0; h < C::kGL; ++h)
                  part[h] = __ffma2_rn(qf[h][c * (C::kVec / 2) + i], kf[i], part[h]);
            }
          }
#pragma unroll
          for (int h = 0; h < C::kGL; ++h) sc[b][h] = part[h].x + part[h].y;
        }
        // the batch's V words, loaded now (row index clamped into the unit;
        // the P.V of a token past ntok is skipped) so that their latency
        // overlaps the score reduction
        uint4 vraw[C::kPreV ? C::kBatch : 1][C::kPreV ? C::kChunks : 1];
        if constexpr (C::kPreV) {
#pragma unroll
          for (int b = 0; b < C::kBatch; ++b) {
            const int t = sub + WH * (tg + C::kTg * (i0 + b));
            const int tl = t < tpu ? t : tpu - 1;
            const T* vrow = vbase + (tl * HKV + g) * D;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              vraw[b][c] = *reinterpret_cast<const uint4*>(vrow + (kl + C::kLpt * c) * C::kVec);
          }
        }
        if constexpr (C::kRS) {
          // Reduce-scatter over the kLpt lanes of a (token slot, head group):
          // scores are laid out head-major (j = h * kBatch + b); each halving
          // exchange keeps one half, so lane kl ends with the complete scores
          // j = kl * kR + i, i < kR, all of head own_h.
          float v[C::kN];
#pragma unroll
          for (int h = 0; h < C::kGL; ++h)
#pragma unroll
            for (int b = 0; b < C::kBatch; ++b) v[h * C::kBatch + b] = sc[b][h];
#pragma unroll
          for (int n = C::kN, off = C::kLpt / 2; off >= 1; n >>= 1, off >>= 1) {
            const bool upper = (kl & off) != 0;
#pragma unroll
            for (int i = 0; i < n / 2; ++i) {
              const float send = upper ? v[i] : v[i + n / 2];
              const float keep = upper ? v[i + n / 2] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
          }
          float m_own = m[0];
#pragma unroll
          for (int h = 1; h < C::kGL; ++h)
            if (own_h == h) m_own = m[h];
          // The running max moves only when a score exceeds it by more than
          // 8 (rare after a sequence's first batch): each lane tests its own
          // scores, and only then does the warp find every head's batch max
          // and rescale, so the common path has no max exchange.
          bool over = false;
#pragma unroll
          for (int i = 0; i < C::kR; ++i) {
            const int t = sub + WH * (tg + C::kTg * (i0 + own_b + i));
            over |= (full || t < ntok) && v[i] > m_own + kRescaleThreshold;
          }
          if (__any_sync(0xffffffffu, over)) {
            float mo = -INFINITY;
#pragma unroll
            for (int i = 0; i < C::kR; ++i) {
              const int t = sub + WH * (tg + C::kTg * (i0 + own_b + i));
              if (full || t < ntok) mo = fmaxf(mo, v[i]);
            }
#pragma unroll
            for (int off = 1; off < C::kLh; off <<= 1)
              mo = fmaxf(mo, __shfl_xor_sync(0xffffffffu, mo, off));
#pragma unroll
            for (int h = 0; h < C::kGL; ++h) {
              const float mx = __shfl_sync(0xffffffffu, mo, base + h * C::kLh);
              const float mn = mx > m[h] + kRescaleThreshold ? mx : m[h];
              const float a = merge_factor(m[h], mn);
              if (own_h == h) l_own *= a;
#pragma unroll
              for (int i = 0; i < C::kPairs; ++i)
                acc[h][i] = make_float2(acc[h][i].x * a, acc[h][i].y * a);
              m[h] = mn;
            }
            m_own = m[0];
#pragma unroll
            for (int h = 1; h < C::kGL; ++h)
              if (own_h == h) m_own = m[h];
          }
          // weights of the lane's own scores, then every lane gathers the
          // weights of all (token, head) pairs it applies to V
          float w_own[C::kR];
#pragma unroll
          for (int i = 0; i < C::kR; ++i) {
            const int t = sub + WH * (tg + C::kTg * (i0 + own_b + i));
            w_own[i] = (full || t < ntok) ? fast_exp2(v[i] - m_own) : 0.f;
            l_own += w_own[i];
          }
#pragma unroll
          for (int h = 0; h < C::kGL; ++h)
#pragma unroll
            for (int b = 0; b < C::kBatch; ++b) {
              const int j = h * C::kBatch + b;
              sc[b][h] = __shfl_sync(0xffffffffu, w_own[j % C::kR], base + j / C::kR);
            }
        } else {
          // complete the dot products across the lanes sharing a (token, head group)
  #pragma unroll
          for (int off = C::kLpt / 2; off >= 1; off >>= 1)
  #pragma unroll
            for (int b = 0; b < C::kBatch; ++b)
  #pragma unroll
              for (int h = 0; h < C::kGL; ++h) sc[b][h] += __shfl_xor_sync(0xffffffffu, sc[b][h], off);
          // online softmax (lazy max, warp-uniform rescale decision)
          float mx[C::kGL];
          bool need = false;
  #pragma unroll
          for (int h = 0; h < C::kGL; ++h) {
            mx[h] = -INFINITY;
  #pragma unroll
            for (int b = 0; b < C::kBatch; ++b) {
              const int t = sub + WH * (tg + C::kTg * (i0 + b));
              if (full || t < ntok) mx[h] = fmaxf(mx[h], sc[b][h]);
            }
            need |= mx[h] > m[h] + kRescaleThreshold;
          }
          if (__any_sync(0xffffffffu, need)) {
  #pragma unroll
            for (int h = 0; h < C::kGL; ++h) {
              const float mn = mx[h] > m[h] + kRescaleThreshold ? mx[h] : m[h];
              const float a = merge_factor(m[h], mn);
              l[h] *= a;
  #pragma unroll
              for (int i = 0; i < C::kPairs; ++i)
                acc[h][i] = make_float2(acc[h][i].x * a, acc[h][i].y * a);
              m[h] = mn;
            }
          }
  #pragma unroll
          for (int b = 0; b < C::kBatch; ++b) {
            const int t = sub + WH * (tg + C::kTg * (i0 + b));
            const bool valid = full || t < ntok;
  #pragma unroll
            for (int h = 0; h < C::kGL; ++h) {
              const float w = valid ? fast_exp2(sc[b][h] - m[h]) : 0.f;
              sc[b][h] = w;
              l[h] += w;
            }
          }
        }
        // P.V
#pragma unroll
        for (int b = 0; b < C::kBatch; ++b) {
          const int t = sub + WH * (tg + C::kTg * (i0 + b));
          if (full || t < ntok) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              float2 vf[C::kVec / 2];
              if constexpr (C::kPreV) {
                unpack_pairs<T>(vraw[b][c], vf);
              } else {
                load_pairs(vbase + (t * HKV + g) * D + (kl + C::kLpt * c) * C::kVec, vf);
              }
#pragma unroll
              for (int h = 0; h < C::kGL; ++h) {
                const float2 w2 = make_float2(sc[b][h], sc[b][h]);
#pragma unroll
                for (int i = 0; i < C::kVec / 2; ++i)
                  acc[h][c * (C::kVec / 2) + i] = __ffma2_rn(w2, vf[i], acc[h][c * (C::kVec / 2) + i]);
              }
            }
          }
        }
      }
      // stage consumed by this warp; the last warp to finish refills it
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        const int prev = atomicAdd(&done[st], 1);
        if (prev == kWarps - 1) {
          done[st] = 0;
          __threadfence_block();
          if (u + L.stages < n_units) issue(u + L.stages, st, false);
        }
      }
      if (++st_c == L.stages) {
        st_c = 0;
        ph_c ^= 1;
      }
    }
    if (!ok) break;

    // ------------------------------------------------------------ finish s
    // 0. reduce-scatter: each head's sum is split over its kLh lanes
    if constexpr (C::kRS) {
#pragma unroll
      for (int off = 1; off < C::kLh; off <<= 1) l_own += __shfl_xor_sync(0xffffffffu, l_own, off);
#pragma unroll
      for (int h = 0; h < C::kGL; ++h) l[h] = __shfl_sync(0xffffffffu, l_own, base + h * C::kLh);
    }
    // 1. merge the token slots of the warp (lanes with equal head group and kl)
#pragma unroll
    for (int off = C::kLanesTok; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < C::kGL; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float lo_ = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float mn = fmaxf(m[h], mo);
        const float a = merge_factor(m[h], mn);
        const float b = merge_factor(mo, mn);
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
    // 2. merge the warps that share a KV head through shared memory; the hand
    //    over is ordered by two mbarriers per KV head (bounded waits)
    if constexpr (WH > 1) {
      const uint32_t ph = static_cast<uint32_t>(merges & 1);
      float* slot_base = merge + g * (WH - 1) * G * (D + 2);
      if (sub > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&merge_empty[g], ph ^ 1u));
        if (ok && tg == 0) {
          float* slot = slot_base + (sub - 1) * G * (D + 2);
#pragma unroll
          for (int h = 0; h < C::kGL; ++h) {
            float* hs = slot + (hg * C::kGL + h) * (D + 2);
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&merge_full[g]);
      } else {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&merge_full[g], ph));
        if (ok) {
          for (int w2 = 1; w2 < WH; ++w2) {
            const float* slot = slot_base + (w2 - 1) * G * (D + 2);
#pragma unroll
            for (int h = 0; h < C::kGL; ++h) {
              const float* hs = slot + (hg * C::kGL + h) * (D + 2);
              const float mo = hs[D], lo_ = hs[D + 1];
              const float mn = fmaxf(m[h], mo);
              const float a = merge_factor(m[h], mn);
              const float b = merge_factor(mo, mn);
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&merge_empty[g]);
      }
      ++merges;
      if (!ok) break;
    }
    // 3. write: the final row when this CTA saw the whole sequence, else a partial
    if (sub == 0 && tg == 0) {
      if (whole && !(has_pre && p.defer_prefix)) {
        T* orow = static_cast<T*>(p.out) + (static_cast<int64_t>(row) * p.hq + head0) * D;
        bool pre_poisoned[C::kGL];
#pragma unroll
        for (int h = 0; h < C::kGL; ++h) pre_poisoned[h] = false;
        if (has_pre) {
          // fold in the shared-prefix partial of this sequence
#pragma unroll
          for (int h = 0; h < C::kGL; ++h) {
            const int64_t idx = static_cast<int64_t>(s) * p.hq + head0 + h;
            const float2 pml = p.pre_ml[idx];
            pre_poisoned[h] = pml.y < 0.f;
            const float mn = fmaxf(m[h], pml.x);
            const float a = merge_factor(m[h], mn), b = merge_factor(pml.x, mn);
            l[h] = l[h] * a + pml.y * b;
            const float* prow = p.pre_acc + idx * D;
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
              for (int i = 0; i < C::kVec / 2; ++i) {
                const int dim = (kl + C::kLpt * c) * C::kVec + 2 * i;
                const float2 pv = *reinterpret_cast<const float2*>(prow + dim);
                float2& r = acc[h][c * (C::kVec / 2) + i];
                r = make_float2(r.x * a + pv.x * b, r.y * a + pv.y * b);
              }
            m[h] = mn;
          }
        }
#pragma unroll
        for (int h = 0; h < C::kGL; ++h) {
          const float inv = (poisoned || pre_poisoned[h]) ? 0.f : 1.f / l[h];
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
        for (int h = 0; h < C::kGL; ++h) {
          const int hh = head0 + h;
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
  if (!ok && lane == 0) status_or(p.d_status, PA_STATUS_TIMEOUT);
}

// Merge the partials of sequences that straddle CTAs: o = sum_c a_c acc_c /
// sum_c a_c l_c with a_c = 2^(m_c - max_c m_c). One warp per (sequence, kHpw
// heads), eight per CTA: the sequence's lookups (record, block range, slots)
// are done once for its heads, and the partials of every head and of four
// CTAs at a time are loaded before any is used, so their latencies overlap.
// kHpw = 1 for small batches (then every row of the batch is read at once),
// more for large ones (fewer warps, fewer waves).
template <typename T, int D, int kHpw>
__global__ void __launch_bounds__(256) decode_reduce_kernel(const DecodeParams p, int grid) {
  pdl_wait_primary();
  constexpr int kPer = D / 32;  // elements per lane
  const int hgroups = p.hq / kHpw;
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (item >= p.num_seqs * hgroups) return;
  const int s = item / hgroups, h0 = (item % hgroups) * kHpw;
  const int lane = threadIdx.x & 31;
  // cascade decode: these rows' prefix partials, loaded first (their
  // addresses depend on nothing else, and are in bounds for every row) so
  // that their latency overlaps the lookups below; used only with a prefix
  float2 pml[kHpw];
  float pacc[kHpw][kPer];
#pragma unroll
  for (int q = 0; q < kHpw; ++q) pml[q] = make_float2(-INFINITY, 0.f);
  if (p.cu_groups != nullptr) {
#pragma unroll
    for (int q = 0; q < kHpw; ++q) {
      const int64_t idx = static_cast<int64_t>(s) * p.hq + h0 + q;
      pml[q] = p.pre_ml[idx];
      const float* src = p.pre_acc + idx * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 x = *reinterpret_cast<const float2*>(src + e);
        pacc[q][e] = x.x;
        pacc[q][e + 1] = x.y;
      }
    }
  }
  // the entry holding s (members ea .. ea + ek - 1; s alone without sibling
  // groups) and whether s has a first-level prefix partial, from the decode
  // kernel's per-sequence record in a cascade call
  int ea = s, ek = 1;
  bool has_pre = false;
  if (p.ws_rec != nullptr) {
    const uint32_t rec = p.ws_rec[s];
    if (!((rec >> 9) & 1u)) return;  // bad lengths: zeroed by the decode kernel
    ea = s - static_cast<int>(rec & 15u);
    ek = static_cast<int>((rec >> 4) & 31u);
    has_pre = (rec >> 10) & 1u;
  }
  const int* prefix = p.ws_prefix;
  const int64_t B = prefix[p.num_seqs];
  const int64_t a0 = prefix[ea], a1 = prefix[ea + ek];
  // CTA c covers blocks [c*B/grid, (c+1)*B/grid)
  int64_t c_first = 0, c_last = -1;  // no CTA partials when the suffix is empty
  if (a1 > a0) {
    c_first = cta_of_block(a0, B, grid);
    c_last = cta_of_block(a1 - 1, B, grid);
    // one CTA saw the whole entry: it wrote the final row, unless the
    // prefix fold was left to this kernel
    if (c_first == c_last && !(p.defer_prefix && has_pre)) return;
  } else if (!has_pre) {
    return;  // not a decode sequence, zeroed by the decode kernel, or nothing to merge
  }
  float m[kHpw], l[kHpw];
  float acc[kHpw][kPer];
#pragma unroll
  for (int q = 0; q < kHpw; ++q) {
    m[q] = -INFINITY;
    l[q] = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[q][e] = 0.f;
  }
  bool poisoned = false;
  // with at least as many blocks as CTAs no CTA range is empty: skip the test
  const bool all_nonempty = B >= grid;
  // this member's partial of CTA c sits at slot0 + c (see the decode kernel)
  const int64_t slot0 = ea + c_first * p.sib_m + static_cast<int64_t>(s - ea) * (c_last - c_first + 1) -
                        c_first;
  constexpr int kC = kHpw > 1 ? 1 : 4;  // CTAs per batch of loads (registers: two CTAs per SM at kHpw 4)
  for (int64_t c0 = c_first; c0 <= c_last; c0 += kC) {
    float2 ml[kHpw][kC];
    float v[kHpw][kC][kPer];
    bool use[kC];
#pragma unroll
    for (int j = 0; j < kC; ++j) {
      const int64_t c = c0 + j;
      use[j] = c <= c_last && (all_nonempty || c * B / grid != (c + 1) * B / grid);
      if (use[j] && (slot0 + c < 0 || slot0 + c >= p.num_slots)) {
        use[j] = false;  // only with inconsistent sibling bounds
        poisoned = true;
      }
      if (use[j]) {
#pragma unroll
        for (int q = 0; q < kHpw; ++q) {
          ml[q][j] = p.ws_ml[(slot0 + c) * p.hq + h0 + q];
          const float* src = p.ws_acc + ((slot0 + c) * p.hq + h0 + q) * D + lane * kPer;
#pragma unroll
          for (int e = 0; e < kPer; e += 2) {
            const float2 x = *reinterpret_cast<const float2*>(src + e);
            v[q][j][e] = x.x;
            v[q][j][e + 1] = x.y;
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kC; ++j) {
      if (!use[j]) continue;
#pragma unroll
      for (int q = 0; q < kHpw; ++q) {
        poisoned |= ml[q][j].y < 0.f;
        const float mn = fmaxf(m[q], ml[q][j].x);
        const float a = merge_factor(m[q], mn), b = merge_factor(ml[q][j].x, mn);
        l[q] = l[q] * a + ml[q][j].y * b;
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[q][e] = acc[q][e] * a + v[q][j][e] * b;
        m[q] = mn;
      }
    }
  }
  // a poisoned partial (a bad block) zeroes the whole row: one poisoned
  // head's partial means its CTA met the block for every head of the sequence
#pragma unroll
  for (int q = 0; q < kHpw; ++q) {
    bool pois = poisoned;
    if (has_pre) {
      pois |= pml[q].y < 0.f;
      const float mn = fmaxf(m[q], pml[q].x);
      const float a = merge_factor(m[q], mn), b = merge_factor(pml[q].x, mn);
      l[q] = l[q] * a + pml[q].y * b;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[q][e] = acc[q][e] * a + pacc[q][e] * b;
    }
    const float inv = pois ? 0.f : 1.f / l[q];
    T* dst = static_cast<T*>(p.out) + (static_cast<int64_t>(query_row(p, s)) * p.hq + h0 + q) * D +
             lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) dst[e] = from_float<T>(acc[q][e] * inv);
  }
}

template <typename T, int D, int G, int WH>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int hkv = kWarps / WH;
  const int elt = sizeof(T);
  const int token_bytes = hkv * D * elt;
  // tokens of one block moved per stage: whole blocks when a K+V block fits 64 KB
  int tpu = kBlockSize;
  while (tpu > 4 && 2 * tpu * token_bytes > 64 * 1024) tpu /= 2;
  const int smem_limit = 227 * 1024 - 1024;  // leave room for static shared memory
  // sibling entries need the tensor-core path (their members share one MMA
  // tile); elsewhere every sequence is walked on its own, which gives the
  // same attention
  const bool sib = Cfg<T, D, G, WH>::kMma && a.cu_sib != nullptr && a.num_sib > 0;
  // a cascade call stages its per-sequence inputs in shared memory when they
  // fit beside the stages (they are read from global memory otherwise)
  const bool cascade = a.cu_groups != nullptr || sib;
  const int meta_ints = cascade ? a.num_seqs + (a.num_groups > 0 ? 2 * a.num_groups + 1 : 0) +
                                      (sib ? 2 * a.num_sib + 1 : 0)
                                : 0;
  SmemLayout L = make_layout(4, tpu, hkv, D, elt, WH, G, a.num_seqs, 0, false);
  if (L.total > smem_limit) L = make_layout(3, tpu, hkv, D, elt, WH, G, a.num_seqs, 0, false);
  if (L.total > smem_limit) L = make_layout(2, tpu, hkv, D, elt, WH, G, a.num_seqs, 0, false);
  if (L.total > smem_limit) return cudaErrorInvalidValue;
  // beside the stages, for a cascade call and when they fit: its staged
  // metadata and the per-sequence facts, else the facts alone (a plain
  // decode's prologue is shorter without them)
  if (cascade) {
    for (const int m : {meta_ints, 0}) {
      const SmemLayout Li = make_layout(L.stages, tpu, hkv, D, elt, WH, G, a.num_seqs, m, true);
      if (Li.total <= smem_limit) {
        L = Li;
        break;
      }
    }
  }

  int grid = a.grid_override > 0 ? a.grid_override : device_sm_count();
  grid = std::min(grid, kMaxDecodeCtas);
  const int sib_m = sib ? 16 / G : 1;
  const size_t slots = a.ws_slots > 0 ? a.ws_slots : static_cast<size_t>(kMaxDecodeCtas) + a.num_seqs;
  // partial slots used: at most num_seqs + sib_m * grid
  if (static_cast<size_t>(a.num_seqs) + static_cast<size_t>(sib_m) * grid > slots)
    return cudaErrorInvalidValue;

  DecodeParams p;
  p.k_pool = static_cast<const char*>(a.pool.k);
  p.v_pool = static_cast<const char*>(a.pool.v);
  p.num_blocks = a.pool.num_blocks;
  p.hkv = hkv;
  p.hq = a.num_q_heads;
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
  const size_t prefix_bytes = align_up_sz((a.num_seqs + 1) * 4, 256);
  p.ws_prefix = reinterpret_cast<int*>(ws);
  p.ws_ml = reinterpret_cast<float2*>(ws + prefix_bytes);
  p.ws_acc = reinterpret_cast<float*>(ws + prefix_bytes + align_up_sz(slots * a.num_q_heads * 8, 256));
  p.d_status = a.d_status;
  p.L = L;
  p.cu_groups = a.cu_groups;
  p.prefix_lens = a.prefix_lens;
  p.num_groups = a.num_groups;
  p.pre_ml = static_cast<const float2*>(a.pre_ml);
  p.pre_acc = static_cast<const float*>(a.pre_acc);
  p.defer_prefix = a.defer_prefix;
  p.cu_sib = sib ? a.cu_sib : nullptr;
  p.shared_lens = sib ? a.shared_lens : nullptr;
  p.num_sib = sib ? a.num_sib : 0;
  p.sib_m = sib_m;
  p.num_slots = static_cast<int64_t>(slots);
  p.ws_rec = cascade ? static_cast<uint32_t*>(a.ws_rec) : nullptr;
  if constexpr (Cfg<T, D, G, WH>::kMma) {
    if (!make_tmap_pool_heads(&p.tm_k, a.pool.k, D, hkv, static_cast<uint64_t>(a.pool.num_blocks)) ||
        !make_tmap_pool_heads(&p.tm_v, a.pool.v, D, hkv, static_cast<uint64_t>(a.pool.num_blocks)))
      return cudaErrorInvalidValue;
  }

  auto kern = decode_kernel<T, D, G, WH, false>;
  if constexpr (Cfg<T, D, G, WH>::kMma) {
    if (sib) kern = decode_kernel<T, D, G, WH, true>;
  }
  if (a.launch_part != 2) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, L.total, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (a.launch_part == 1) return cudaSuccess;  // the caller launches the merge later

  // merge kernel, launched with programmatic stream serialization so its
  // launch overlaps the decode kernel's tail (it waits with griddepcontrol.wait);
  // launched on its own (after a join of streams) it needs no such overlap
  // one warp per (sequence, head) while the rows fit in one wave of warps
  // (64 per SM), else per (sequence, 4 heads)
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  const int hpw = (a.num_q_heads % 4 == 0 && rows > 64LL * device_sm_count()) ? 4 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows / hpw + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.launch_part == 2 ? 0 : 1;
  if (hpw == 4) return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<T, D, 4>, p, grid);
  return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<T, D, 1>, p, grid);
}

template <typename T, int D, int G>
cudaError_t dispatch_wh(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.pool.num_kv_heads) {
    case 8: return launch_typed<T, D, G, 1>(a, stream);
    case 4: return launch_typed<T, D, G, 2>(a, stream);
    case 2: return launch_typed<T, D, G, 4>(a, stream);
    case 1: return launch_typed<T, D, G, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Dispatch on the GQA group and the number of KV heads for one (dtype, head_dim).
template <typename T, int D>
cudaError_t dispatch_decode_d(const DecodeArgs& a, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return dispatch_wh<T, D, 1>(a, stream);
    case 2: return dispatch_wh<T, D, 2>(a, stream);
    case 4: return dispatch_wh<T, D, 4>(a, stream);
    case 8: return dispatch_wh<T, D, 8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
