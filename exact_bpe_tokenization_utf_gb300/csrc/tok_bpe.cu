// Per-fragment BPE, E ("TokTier: exact stateful tokenization for agentic LLM
// serving", Section 4.2): every fragment is encoded on its own by merging the
// lowest-rank adjacent pair (leftmost on ties) until no adjacent pair is a
// merge.  The pages tier fragments by length (one thread, one warp, one
// block); the tiers here are this library's own:
//
//   thread tier (<= 16 bytes)  the rule itself, symbols in registers
//   warp tier   (<= 256 bytes) the sweep engine below, arrays in shared memory
//   CTA tier    (longer)       the sweep engine, arrays in global memory
//
// Sweep engine.  Let k be the rank of pair j = (s_j, s_{j+1}).  When every
// merge that uses a token comes after every merge that produces it (the
// vocabulary is "monotone", checked at load), the textbook loop merges in
// non-decreasing rank order, and pair j is merged exactly as it stands unless
// s_j or s_{j+1} is absorbed by a lower-rank merge first.  That can only be
//   - pair j-1 or j+1 having a lower rank now, or
//   - a token Y grown from a lower-rank pair further left that ends at s_{j-1}
//     and then merges with s_j, which needs |Y| <= the longest left operand of
//     any merge with right operand s_j (and the mirror image on the right):
//     every merge inside the window between that lower-rank pair and j must
//     involve the growing token, so Y covers all symbols in between.
// A pair that none of these can reach is "safe"; equal-rank pairs that
// overlap (runs of one symbol x with the merge (x,x)) pair up from the left
// end of the run, which must itself be safe.  Every sweep merges all safe
// pairs at once; the leftmost minimum pair is always safe, so each sweep makes
// progress, and the result equals the textbook loop.  For other vocabularies
// the engine falls back to merging only the leftmost minimum pair per sweep,
// which is the textbook loop itself.
#include "tok_common.cuh"

namespace tokgb {

constexpr unsigned long long KR_NONE = ~0ull;
constexpr unsigned long long KR_NEED = ~0ull - 1ull;  // key to be looked up
constexpr uint32_t SYM_MASK = 0xFFFFFu;

// ---------------------------------------------------------------------------
// thread tier

__device__ __forceinline__ void bpe_thread(const DevVocab& V, const int32_t* s_byte_id, const uint8_t* text,
                                           long long a, int len, int32_t* sid, uint8_t* tstart) {
  // s: symbol (bits 0-19) | byte length (bits 20-27); r: rank; x: result
  uint32_t s[SHORT_MAX], r[SHORT_MAX], x[SHORT_MAX];
#pragma unroll
  for (int k = 0; k < SHORT_MAX; ++k) s[k] = k < len ? ((uint32_t)s_byte_id[text[a + k]] | (1u << 20)) : 0u;
#pragma unroll
  for (int k = 0; k < SHORT_MAX; ++k) {
    r[k] = NO_RANK;
    x[k] = 0;
    if (k + 1 < len) {
      const unsigned long long e = merge_lookup(V, s[k] & SYM_MASK, s[k + 1] & SYM_MASK);
      r[k] = kr_rank(e);
      x[k] = kr_result(e);
    }
  }
  int m = len;
  for (int it = 0; it < SHORT_MAX; ++it) {
    uint32_t best = r[0];
    int j = 0;
#pragma unroll
    for (int k = 1; k < SHORT_MAX - 1; ++k)
      if (r[k] < best) { best = r[k]; j = k; }
    if (best == NO_RANK) break;
    uint32_t sj = 0, sj1 = 0, xj = 0;
#pragma unroll
    for (int k = 0; k < SHORT_MAX; ++k) {
      if (k == j) { sj = s[k]; xj = x[k]; }
      if (k == j + 1) sj1 = s[k];
    }
    const uint32_t merged = xj | ((((sj >> 20) + (sj1 >> 20))) << 20);
#pragma unroll
    for (int k = 0; k < SHORT_MAX; ++k) {
      const uint32_t nxt_s = k + 1 < SHORT_MAX ? s[k + 1] : 0u;
      const uint32_t nxt_r = k + 1 < SHORT_MAX ? r[k + 1] : NO_RANK;
      const uint32_t nxt_x = k + 1 < SHORT_MAX ? x[k + 1] : 0u;
      if (k == j) s[k] = merged;
      else if (k > j) { s[k] = nxt_s; r[k] = nxt_r; x[k] = nxt_x; }
    }
    --m;
    // neighbours of the new symbol
    uint32_t left = 0, right = 0;
#pragma unroll
    for (int k = 0; k < SHORT_MAX; ++k) {
      if (k == j - 1) left = s[k];
      if (k == j + 1) right = s[k];
    }
    unsigned long long el = KR_NONE, er = KR_NONE;
    if (j > 0) el = merge_lookup(V, left & SYM_MASK, merged & SYM_MASK);
    if (j + 1 < m) er = merge_lookup(V, merged & SYM_MASK, right & SYM_MASK);
#pragma unroll
    for (int k = 0; k < SHORT_MAX; ++k) {
      if (k == j - 1) { r[k] = kr_rank(el); x[k] = kr_result(el); }
      if (k == j) { r[k] = kr_rank(er); x[k] = kr_result(er); }
    }
  }
  // outputs: token id at each token's first byte, token-start flags
  uint32_t starts = 0;
  int off = 0;
#pragma unroll
  for (int k = 0; k < SHORT_MAX; ++k) {
    if (k < m) {
      sid[a + off] = (int32_t)(s[k] & SYM_MASK);
      starts |= 1u << off;
      off += (int)(s[k] >> 20);
    }
  }
#pragma unroll
  for (int k = 0; k < SHORT_MAX; ++k)
    if (k < len) tstart[a + k] = (uint8_t)((starts >> k) & 1u);
}

// K3: enumerate the fragments that start in this CTA's 1 KiB range, encode
// the short ones, queue the others
__global__ void __launch_bounds__(BPE_THREADS) k_bpe_short(Call c, Workspace ws, DevVocab V) {
  constexpr int WORDS = BPE_CHUNK / 32;
  constexpr int EXT = MED_MAX / 32 + 2;  // words scanned past the range for the last fragment's end
  __shared__ uint32_t words[WORDS];
  __shared__ uint16_t starts[BPE_CHUNK + 1];
  __shared__ int32_t s_byte_id[256];
  __shared__ int wsum[BPE_THREADS / 32];
  __shared__ long long s_last_end;
  const int tid = threadIdx.x;
  const long long r0 = (long long)blockIdx.x * BPE_CHUNK;
  const long long r1 = min(r0 + BPE_CHUNK, c.n);
  s_byte_id[tid] = V.byte_id[tid];
  if (tid < WORDS) words[tid] = (r0 + tid * 32 < c.n) ? ws.pstart[(r0 >> 5) + tid] : 0u;
  if (tid == 0) {
    // end of the last fragment: next start at or after r1, the text end, or unknown
    long long e = -1;
    if (r1 >= c.n) e = c.n;
    else {
      for (int q = 0; q < EXT && e < 0; ++q) {
        const long long wi = (r1 >> 5) + q;
        if (wi * 32 >= c.n) { e = c.n; break; }
        uint32_t wv = ws.pstart[wi];
        if (q == 0) wv &= ~0u << (r1 & 31);
        if (wv) e = min(wi * 32 + __ffs(wv) - 1, c.n);
      }
    }
    s_last_end = e;
  }
  __syncthreads();
  // positions of starts: thread t scans bits [4t, 4t+4)
  const uint32_t nib = (words[tid >> 3] >> ((tid & 7) * 4)) & 0xFu;
  const int cnt = __popc(nib);
  // block exclusive sum
  const int lane = tid & 31, warp = tid >> 5;
  int inc = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int wpre = 0, total = 0;
  for (int k = 0; k < BPE_THREADS / 32; ++k) {
    if (k < warp) wpre += wsum[k];
    total += wsum[k];
  }
  int pos = wpre + inc - cnt;
  for (int q = 0; q < 4; ++q)
    if ((nib >> q) & 1u) starts[pos++] = (uint16_t)(tid * 4 + q);
  __syncthreads();
  for (int k = tid; k < total; k += BPE_THREADS) {
    const long long a = r0 + starts[k];
    const long long e = (k + 1 < total) ? r0 + starts[k + 1] : s_last_end;
    const long long len = e < 0 ? -1 : e - a;
    if (len >= 1 && len <= SHORT_MAX) {
      bpe_thread(V, s_byte_id, c.text, a, (int)len, ws.sid, ws.tstart);
    } else if (len >= 1 && len <= MED_MAX) {
      const uint32_t q = atomicAdd(&ws.st->med_count, 1u);
      ws.medq[q] = Frag{a, len};
    } else {
      const uint32_t q = atomicAdd(&ws.st->long_count, 1u);
      ws.longq[q] = Frag{a, len};
    }
  }
}

// ---------------------------------------------------------------------------
// groups for the sweep engine

struct WarpGroup {
  __device__ int rank() const { return threadIdx.x & 31; }
  __device__ int size() const { return 32; }
  __device__ void sync() const { __syncwarp(); }
  __device__ bool any(bool p) const { return __any_sync(0xffffffffu, p); }
  __device__ int excl_sum(int v, int* total) const {
    const int lane = threadIdx.x & 31;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += o;
    }
    *total = __shfl_sync(0xffffffffu, inc, 31);
    return inc - v;
  }
  __device__ int excl_max(int v) const {
    const int lane = threadIdx.x & 31;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc = max(inc, o);
    }
    const int ex = __shfl_up_sync(0xffffffffu, inc, 1);
    return lane == 0 ? -1 : ex;
  }
  __device__ unsigned long long min_u64(unsigned long long v) const {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
      v = o < v ? o : v;
    }
    return v;
  }
};

// whole-CTA group; `sh` is shared scratch of at least 2 * (blockDim/32) + 2 words
struct BlockGroup {
  long long* sh;
  __device__ int rank() const { return threadIdx.x; }
  __device__ int size() const { return blockDim.x; }
  __device__ void sync() const { __syncthreads(); }
  __device__ bool any(bool p) const { return __syncthreads_or(p) != 0; }
  __device__ int excl_sum(int v, int* total) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += o;
    }
    __syncthreads();
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    long long pre = 0, tot = 0;
    for (int k = 0; k < nw; ++k) {
      if (k < warp) pre += sh[k];
      tot += sh[k];
    }
    *total = (int)tot;
    __syncthreads();
    return (int)pre + inc - v;
  }
  __device__ int excl_max(int v) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc = max(inc, o);
    }
    __syncthreads();
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    int pre = -1;
    for (int k = 0; k < warp; ++k) pre = max(pre, (int)sh[k]);
    const int ex = __shfl_up_sync(0xffffffffu, inc, 1);
    __syncthreads();
    return lane == 0 ? pre : max(pre, ex);
  }
  __device__ unsigned long long min_u64(unsigned long long v) const {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
      v = o < v ? o : v;
    }
    __syncthreads();
    if (lane == 0) sh[warp] = (long long)v;
    __syncthreads();
    unsigned long long r = ~0ull;
    for (int k = 0; k < nw; ++k) {
      const unsigned long long o = (unsigned long long)sh[k];
      r = o < r ? o : r;
    }
    __syncthreads();
    return r;
  }
};

struct EngineArrays {
  uint32_t* sym[2];
  uint16_t* len[2];
  unsigned long long* kr[2];
  uint8_t* fl;   // bit 0: pair merges this sweep
  int32_t* rs;   // start of the run of equal-rank pairs containing this pair
};

// Is pair i (rank k) safe to merge now?  See the file comment.
__device__ __forceinline__ bool pair_safe(const DevVocab& V, const uint32_t* S, const uint16_t* L,
                                          const unsigned long long* K, const int32_t* rs, int m, int i,
                                          uint32_t k) {
  const int u = rs[i];
  if ((i - u) & 1) return false;  // overlapping equal pairs pair up from the run start
  if (u > 0) {
    if (kr_rank(K[u - 1]) < k) return false;
    const int lim = V.max_left[S[u]];
    int cum = L[u - 1];
    for (int q = u - 2; q >= 0; --q) {
      cum += L[q];
      if (cum > lim) break;
      if (kr_rank(K[q]) < k) return false;
    }
  }
  if (i + 1 < m - 1) {
    if (kr_rank(K[i + 1]) < k) return false;
    const int lim = V.max_right[S[i + 1]];
    int cum = L[i + 2];
    for (int q = i + 2; q < m - 1; ++q) {
      cum += L[q + 1];
      if (cum > lim) break;
      if (kr_rank(K[q]) < k) return false;
    }
  }
  return true;
}

// Encode the fragment text[a .. a+m0) with group g.  Arrays hold >= m0
// elements.  Writes sid / tstart for the fragment's bytes.
template <class G>
__device__ void sweep_engine(const G& g, const DevVocab& V, const uint8_t* text, long long a, int m0,
                             const EngineArrays& A, int32_t* sid, uint8_t* tstart, int32_t* err) {
  const int t = g.rank(), GS = g.size();
  int m = m0;
  for (int i = t; i < m; i += GS) {
    A.sym[0][i] = (uint32_t)V.byte_id[text[a + i]];
    A.len[0][i] = 1;
  }
  g.sync();
  for (int i = t; i < m; i += GS)
    A.kr[0][i] = (i + 1 < m) ? merge_lookup(V, A.sym[0][i], A.sym[0][i + 1]) : KR_NONE;
  g.sync();
  int cur = 0;
  for (int sweep = 0; sweep <= m0; ++sweep) {
    const uint32_t* S = A.sym[cur];
    const uint16_t* L = A.len[cur];
    const unsigned long long* K = A.kr[cur];
    const int np = m - 1;  // pairs
    // 1. run starts of equal-rank pairs, contiguous blocks per thread
    const int E = (np + GS - 1) / GS;
    const int lo = min(t * E, np), hi = min(lo + E, np);
    int last = -1;
    for (int i = lo; i < hi; ++i)
      if (i == 0 || kr_rank(K[i - 1]) != kr_rank(K[i])) last = i;
    int run = g.excl_max(last);
    for (int i = lo; i < hi; ++i) {
      if (i == 0 || kr_rank(K[i - 1]) != kr_rank(K[i])) run = i;
      A.rs[i] = run;
    }
    g.sync();
    // 2. safe pairs
    bool any_pair = false, any_safe = false;
    if (V.monotone) {
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(K[i]);
        uint8_t f = 0;
        if (k != NO_RANK) {
          any_pair = true;
          if (pair_safe(V, S, L, K, A.rs, m, i, k)) { f = 1; any_safe = true; }
        }
        A.fl[i] = f;
      }
    } else {
      unsigned long long best = ~0ull;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(K[i]);
        if (k != NO_RANK) {
          const unsigned long long key = ((unsigned long long)k << 32) | (uint32_t)i;
          best = key < best ? key : best;
        }
      }
      best = g.min_u64(best);
      any_pair = best != ~0ull;
      any_safe = any_pair;
      for (int i = lo; i < hi; ++i) A.fl[i] = (any_pair && (uint32_t)best == (uint32_t)i) ? 1 : 0;
    }
    if (t == 0 && m > 0) A.fl[m - 1] = 0;
    g.sync();
    any_pair = g.any(any_pair);
    any_safe = g.any(any_safe);
    if (!any_pair) break;
    if (!any_safe) {  // cannot happen: the leftmost minimum pair is always safe
      if (t == 0) atomicExch(err, ST_EINTERNAL);
      break;
    }
    // 3. merge and compact into the other buffer
    const int E2 = (m + GS - 1) / GS;
    const int lo2 = min(t * E2, m), hi2 = min(lo2 + E2, m);
    int keep = 0;
    for (int i = lo2; i < hi2; ++i) keep += !(i > 0 && A.fl[i - 1]);
    int newm = 0;
    int p = g.excl_sum(keep, &newm);
    uint32_t* S2 = A.sym[cur ^ 1];
    uint16_t* L2 = A.len[cur ^ 1];
    unsigned long long* K2 = A.kr[cur ^ 1];
    for (int i = lo2; i < hi2; ++i) {
      if (i > 0 && A.fl[i - 1]) continue;  // absorbed into its left neighbour
      const bool mg = A.fl[i] != 0;
      if (mg) {
        S2[p] = kr_result(K[i]);
        L2[p] = (uint16_t)(L[i] + L[i + 1]);
      } else {
        S2[p] = S[i];
        L2[p] = L[i];
      }
      // an unchanged pair keeps its rank; pairs touching a new symbol are looked up
      K2[p] = (!mg && i + 1 < m && !A.fl[i + 1]) ? K[i] : KR_NEED;
      ++p;
    }
    g.sync();
    for (int q = t; q < newm; q += GS) {
      if (q + 1 >= newm) K2[q] = KR_NONE;
      else if (K2[q] == KR_NEED) K2[q] = merge_lookup(V, S2[q], S2[q + 1]);
    }
    g.sync();
    cur ^= 1;
    m = newm;
  }
  // outputs
  const int E3 = (m + GS - 1) / GS;
  const int lo3 = min(t * E3, m), hi3 = min(lo3 + E3, m);
  int bytes = 0;
  for (int i = lo3; i < hi3; ++i) bytes += A.len[cur][i];
  int tot = 0;
  int off = g.excl_sum(bytes, &tot);
  for (int i = lo3; i < hi3; ++i) {
    const int l = A.len[cur][i];
    sid[a + off] = (int32_t)A.sym[cur][i];
    tstart[a + off] = 1;
    for (int q = 1; q < l; ++q) tstart[a + off + q] = 0;
    off += l;
  }
  g.sync();
}

// K4a: warp tier, fragments of 17..256 bytes, arrays in shared memory
struct WarpArrays {
  uint32_t sym[2][MED_MAX];
  unsigned long long kr[2][MED_MAX];
  uint16_t len[2][MED_MAX];
  int32_t rs[MED_MAX];
  uint8_t fl[MED_MAX];
};

__global__ void __launch_bounds__(MED_WARPS * 32) k_bpe_med(Call c, Workspace ws, DevVocab V) {
  __shared__ WarpArrays wa[MED_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpArrays& W = wa[warp];
  EngineArrays A;
  A.sym[0] = W.sym[0]; A.sym[1] = W.sym[1];
  A.len[0] = W.len[0]; A.len[1] = W.len[1];
  A.kr[0] = W.kr[0]; A.kr[1] = W.kr[1];
  A.fl = W.fl; A.rs = W.rs;
  WarpGroup g;
  const uint32_t count = *(volatile uint32_t*)&ws.st->med_count;
  while (true) {
    uint32_t idx = 0;
    if (lane == 0) idx = atomicAdd(&ws.st->med_taken, 1u);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    if (idx >= count) break;
    const Frag f = ws.medq[idx];
    sweep_engine(g, V, c.text, f.start, (int)f.len, A, ws.sid, ws.tstart, &ws.st->code);
  }
}

// K4b: CTA tier, fragments longer than 256 bytes (or of unknown length),
// arrays in global memory at the fragment's byte offsets
__global__ void __launch_bounds__(LONG_THREADS) k_bpe_long(Call c, Workspace ws, DevVocab V) {
  __shared__ long long sh[2 * (LONG_THREADS / 32) + 4];
  __shared__ uint32_t s_idx;
  __shared__ long long s_end;
  BlockGroup g{sh};
  const uint32_t count = *(volatile uint32_t*)&ws.st->long_count;
  while (true) {
    if (threadIdx.x == 0) s_idx = atomicAdd(&ws.st->long_taken, 1u);
    __syncthreads();
    const uint32_t idx = s_idx;
    __syncthreads();
    if (idx >= count) break;
    const Frag f = ws.longq[idx];
    long long len = f.len;
    if (len < 0) {
      // find the next fragment start after f.start (first set bit), bounded by n
      if (threadIdx.x == 0) s_end = c.n;
      __syncthreads();
      const long long w0 = (f.start + 1) >> 5;
      const long long wn = (c.n + 31) >> 5;
      for (long long base = w0; base < wn; base += blockDim.x) {
        const long long wi = base + threadIdx.x;
        if (wi < wn) {
          uint32_t wv = ws.pstart[wi];
          if (wi == w0) wv &= ~0u << ((f.start + 1) & 31);
          if (wv) atomicMin((unsigned long long*)&s_end, (unsigned long long)min(wi * 32 + __ffs(wv) - 1, c.n));
        }
        __syncthreads();
        const long long e = s_end;
        __syncthreads();
        if (e < c.n || base + blockDim.x >= wn) break;
      }
      len = s_end - f.start;
      __syncthreads();
    }
    EngineArrays A;
    for (int b = 0; b < 2; ++b) {
      A.sym[b] = ws.e_sym[b] + f.start;
      A.len[b] = ws.e_len[b] + f.start;
      A.kr[b] = ws.e_kr[b] + f.start;
    }
    A.fl = ws.e_fl + f.start;
    A.rs = ws.e_rs + f.start;
    sweep_engine(g, V, c.text, f.start, (int)len, A, ws.sid, ws.tstart, &ws.st->code);
  }
}

void launch_bpe_short(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s) {
  const long long nb = (c.n + BPE_CHUNK - 1) / BPE_CHUNK;
  k_bpe_short<<<(unsigned)nb, BPE_THREADS, 0, s>>>(c, w, v);
}

void launch_bpe_med(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_med<<<n_sms * 4, MED_WARPS * 32, 0, s>>>(c, w, v);
}

void launch_bpe_long(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_long<<<n_sms, LONG_THREADS, 0, s>>>(c, w, v);
}

}  // namespace tokgb
