// prefill_simt.cu -- chunked-prefill attention on CUDA cores (fp32 path).
//
// A prefill chunk of q_len tokens of sequence s (context ctx, which includes
// the chunk) attends causally over absolute positions: query row i sits at
// position ctx - q_len + i and sees keys 0 .. that position, i.e. everything
// cached by earlier chunks plus the chunk's own tokens up to itself ("Chunked
// Prefill" glossary page: each chunk uses the cached keys and values of all
// earlier chunks plus its own tokens under a causal mask, the mask being
// ones(end - start, end).tril(diagonal = start)). Keys are gathered through
// the block table.
//
// One CTA handles 64 query rows (64 / G tokens x the G query heads of one KV
// head) so each K/V tile is loaded once for the whole GQA group. Keys advance
// one 16-token block at a time; the online softmax runs per row in fp32.
// Tensor cores serve the bf16 path (prefill_tc.cu); this kernel is the fp32
// path and checks the bf16 one.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kRows = 64;
constexpr int kThreads = 256;

struct PrefillSimtParams {
  const char* k_pool;
  const char* v_pool;
  int64_t num_blocks;
  int hkv, hq, group;
  const void* q;
  void* out;
  const int32_t* cu_q_lens;
  int num_seqs;
  int num_rows;
  const int32_t* block_tables;
  int max_blocks;
  const int32_t* context_lens;
  float scale_log2;
  int* d_status;
};

__device__ __forceinline__ int prefill_tiles(const PrefillSimtParams& p, int s, int tq) {
  // a prefill chunk is any sequence with more than one query row this step
  const int q0 = p.cu_q_lens[s], q1 = p.cu_q_lens[s + 1];
  if (q0 < 0 || q1 > p.num_rows || q1 - q0 <= 1) return 0;  // not a (well-formed) chunk
  return (q1 - q0 + tq - 1) / tq;
}

template <int D>
struct SimtSmem {
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kRows * (D + 1);
  static constexpr int kV = kK + kBlockSize * (D + 1);
  static constexpr int kP = kV + kBlockSize * (D + 1);
  static constexpr int kFloats = kP + kRows * (kBlockSize + 1);
  static int bytes(int num_seqs) { return kFloats * 4 + (num_seqs + 1) * 4; }
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillSimtParams p) {
  using L = SimtSmem<D>;
  extern __shared__ __align__(16) float dyn[];
  float(*Qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn + L::kQ);
  float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn + L::kK);
  float(*Vs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn + L::kV);
  float(*Ps)[kBlockSize + 1] = reinterpret_cast<float(*)[kBlockSize + 1]>(dyn + L::kP);
  int* tile_prefix = reinterpret_cast<int*>(dyn + L::kFloats);
  __shared__ float row_m[kRows], row_l[kRows], row_alpha[kRows];
  __shared__ int row_pos[kRows];
  __shared__ int warp_sums[kThreads / 32];
  __shared__ int sh_bad;

  const int tid = threadIdx.x;
  const int G = p.group;
  const int tq = kRows / G;  // tokens per tile
  const int g = blockIdx.y;

  // this CTA's (sequence, tile): scan of per-sequence tile counts
  block_exclusive_scan<kThreads>(
      p.num_seqs, [&](int i) { return prefill_tiles(p, i, tq); }, tile_prefix, warp_sums);
  if (static_cast<int>(blockIdx.x) >= tile_prefix[p.num_seqs]) return;
  const int s = upper_index(tile_prefix, p.num_seqs, blockIdx.x);
  const int tile = blockIdx.x - tile_prefix[s];
  if (tid == 0) sh_bad = 0;
  const int q0 = p.cu_q_lens[s];
  const int q_len = p.cu_q_lens[s + 1] - q0;
  const int ctx = p.context_lens[s];
  const int tok0 = tile * tq;
  const int ntok = min(tq, q_len - tok0);
  const bool bad_len = ctx > p.max_blocks * kBlockSize || q_len > ctx;

  // stage the tile's queries (fp32, log2-domain scaled) and row positions
  for (int i = tid; i < kRows * D; i += kThreads) {
    const int r = i / D, e = i % D;
    const int tok = r / G, hh = r % G;
    float v = 0.f;
    if (tok < ntok && !bad_len) {
      const T* qrow = static_cast<const T*>(p.q) +
                      (static_cast<int64_t>(q0 + tok0 + tok) * p.hq + g * G + hh) * D;
      v = to_float(qrow[e]) * p.scale_log2;
    }
    Qs[r][e] = v;
  }
  if (tid < kRows) {
    const int tok = tid / G;
    row_pos[tid] = tok < ntok ? ctx - q_len + tok0 + tok : -1;
    row_m[tid] = -INFINITY;
    row_l[tid] = 0.f;
  }
  __syncthreads();

  const int r_out = tid / 4, qd = tid % 4;  // P.V ownership: row, quarter of head_dim
  constexpr int kQ = D / 4;
  float acc[kQ];
#pragma unroll
  for (int e = 0; e < kQ; ++e) acc[e] = 0.f;

  const int max_pos = ctx - q_len + tok0 + ntok - 1;
  const int n_kt = bad_len ? 0 : max_pos / kBlockSize + 1;
  const int token_elems = p.hkv * D;
  for (int kt = 0; kt < n_kt; ++kt) {
    const int phys = p.block_tables[static_cast<int64_t>(s) * p.max_blocks + kt];
    if (phys < 0 || phys >= p.num_blocks) {
      if (tid == 0) sh_bad = 1;
      break;
    }
    // load the key/value block of KV head g (zeros past the context)
    for (int i = tid; i < kBlockSize * D; i += kThreads) {
      const int k = i / D, e = i % D;
      const int kp = kt * kBlockSize + k;
      float kv = 0.f, vv = 0.f;
      if (kp < ctx) {
        const int64_t off = (static_cast<int64_t>(phys) * kBlockSize + k) * token_elems + g * D + e;
        kv = to_float(reinterpret_cast<const T*>(p.k_pool)[off]);
        vv = to_float(reinterpret_cast<const T*>(p.v_pool)[off]);
      }
      Ks[k][e] = kv;
      Vs[k][e] = vv;
    }
    __syncthreads();
    // scores: thread -> (row, 4 keys)
    {
      const int r = tid / 4;
      for (int j = 0; j < 4; ++j) {
        const int k = tid % 4 + 4 * j;
        const int kp = kt * kBlockSize + k;
        float dot = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) dot += Qs[r][e] * Ks[k][e];
        Ps[r][k] = (row_pos[r] >= 0 && kp <= row_pos[r]) ? dot : -INFINITY;
      }
    }
    __syncthreads();
    // per-row online softmax update
    if (tid < kRows) {
      const int r = tid;
      float mx = row_m[r];
      for (int k = 0; k < kBlockSize; ++k) mx = fmaxf(mx, Ps[r][k]);
      const float alpha = (row_m[r] == -INFINITY) ? 0.f : exp2f(row_m[r] - mx);
      float lsum = row_l[r] * alpha;
      for (int k = 0; k < kBlockSize; ++k) {
        const float w = (Ps[r][k] == -INFINITY) ? 0.f : exp2f(Ps[r][k] - mx);
        Ps[r][k] = w;
        lsum += w;
      }
      row_m[r] = mx;
      row_l[r] = lsum;
      row_alpha[r] = alpha;
    }
    __syncthreads();
    {
      const float a = row_alpha[r_out];
#pragma unroll
      for (int e = 0; e < kQ; ++e) {
        float o = acc[e] * a;
        for (int k = 0; k < kBlockSize; ++k) o += Ps[r_out][k] * Vs[k][qd * kQ + e];
        acc[e] = o;
      }
    }
    __syncthreads();
  }
  __syncthreads();
  if (tid == 0 && (sh_bad || bad_len))
    status_or(p.d_status, sh_bad ? PA_STATUS_BAD_BLOCK : PA_STATUS_BAD_LENGTH);
  const int tok = r_out / G, hh = r_out % G;
  if (tok < ntok) {
    const bool zero = sh_bad || bad_len;
    const float inv = zero ? 0.f : 1.f / row_l[r_out];
    T* orow = static_cast<T*>(p.out) + (static_cast<int64_t>(q0 + tok0 + tok) * p.hq + g * G + hh) * D;
#pragma unroll
    for (int e = 0; e < kQ; ++e) orow[qd * kQ + e] = from_float<T>(acc[e] * inv);
  }
}

template <typename T>
cudaError_t launch_simt_typed(const PrefillArgs& a, cudaStream_t stream) {
  PrefillSimtParams p;
  p.k_pool = static_cast<const char*>(a.pool.k);
  p.v_pool = static_cast<const char*>(a.pool.v);
  p.num_blocks = a.pool.num_blocks;
  p.hkv = a.pool.num_kv_heads;
  p.hq = a.num_q_heads;
  p.group = a.num_q_heads / a.pool.num_kv_heads;
  p.q = a.q;
  p.out = a.out;
  p.cu_q_lens = a.cu_q_lens;
  p.num_seqs = a.num_seqs;
  p.num_rows = a.num_tokens;
  p.block_tables = a.block_tables;
  p.max_blocks = a.max_blocks_per_seq;
  p.context_lens = a.context_lens;
  p.scale_log2 = a.scale * kLog2e;
  p.d_status = a.d_status;
  const int tq = kRows / p.group;
  const int tiles = (a.num_tokens + tq - 1) / tq + a.num_seqs;  // upper bound
  dim3 grid(tiles, p.hkv);
  auto run = [&](auto kern, int smem) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  };
  switch (a.pool.head_dim) {
    case 64: return run(prefill_simt_kernel<T, 64>, SimtSmem<64>::bytes(a.num_seqs));
    case 128: return run(prefill_simt_kernel<T, 128>, SimtSmem<128>::bytes(a.num_seqs));
    case 256: return run(prefill_simt_kernel<T, 256>, SimtSmem<256>::bytes(a.num_seqs));
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
  if (a.num_tokens == 0 || a.num_seqs == 0) return cudaSuccess;
  if (a.pool.dtype == PA_BF16) return launch_simt_typed<__nv_bfloat16>(a, stream);
  return launch_simt_typed<float>(a, stream);
}

}  // namespace pa
