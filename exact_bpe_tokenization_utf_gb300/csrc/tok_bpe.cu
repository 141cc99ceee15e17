// Per-fragment BPE, E ("TokTier: exact stateful tokenization for agentic LLM
// serving", Section 4.2): every fragment is encoded on its own by merging the
// lowest-rank adjacent pair (leftmost on ties) until no adjacent pair is a
// merge.  The pages tier fragments by length (one thread, one warp, one block
// per fragment); here one CTA encodes all fragments of a 1 KiB chunk at once,
// and only fragments longer than that get a CTA each.
//
// Sweep engine.  The symbols of many fragments sit in one array; the pair
// between two fragments is a "wall" that never merges.  Let k be the rank of
// pair j = (s_j, s_{j+1}).  When every merge that uses a token comes after
// every merge that produces it (the vocabulary is "monotone", checked at
// load), the rule merges in non-decreasing rank order, and pair j is merged
// exactly as it stands unless s_j or s_{j+1} is absorbed by a lower-rank merge
// first.  That can only be
//   - pair j-1 or j+1 having a lower rank now, or
//   - a token Y grown from a lower-rank pair further left that ends at s_{j-1}
//     and then merges with s_j, which needs |Y| <= the longest left operand of
//     any merge whose right operand is s_j (and the mirror image on the
//     right): every merge between that lower-rank pair and j must involve the
//     growing token, so Y covers all symbols in between; a wall stops it.
// A pair none of these can reach is "safe".  Equal-rank pairs that overlap
// (runs of one symbol x with the merge (x,x)) pair up from the left end of
// the run, which must itself be safe.  Every sweep merges all safe pairs; the
// leftmost minimum pair of each fragment is always safe, so every sweep makes
// progress, and the result equals the rule.  For other vocabularies a sweep
// merges only the leftmost minimum pair of the whole array, which is the
// rule itself applied fragment after fragment.
#include "tok_common.cuh"

namespace tokgb {

// pair keys: rank << 32 | result
constexpr uint32_t RANK_NONE = 0xFFFFFFFFu;  // not a merge (may become one when a symbol changes)
constexpr uint32_t RANK_WALL = 0xFFFFFFFEu;  // between fragments, or past the last symbol: never merges
constexpr uint32_t RANK_NEED = 0xFFFFFFFDu;  // to be looked up
constexpr unsigned long long KR_WALL = (unsigned long long)RANK_WALL << 32;
constexpr unsigned long long KR_NEED = (unsigned long long)RANK_NEED << 32;
constexpr uint16_t LEN_MASK = 0x7FFF;        // symbol byte length; bit 15: symbol starts a fragment
constexpr uint16_t FRAG_START = 0x8000;

__device__ __forceinline__ bool mergeable(uint32_t rank) { return rank < RANK_NEED; }

// Is pair i (rank k) safe to merge now?  rs[i] is the first pair of the run
// of equal-rank pairs that contains i.  See the file comment.
template <class RS>
__device__ __forceinline__ bool pair_safe(const DevVocab& V, const uint32_t* S, const uint16_t* L,
                                          const unsigned long long* K, const RS* rs, int m, int i, uint32_t k) {
  const int u = (int)rs[i];
  if ((i - u) & 1) return false;
  if (u > 0) {
    const uint32_t kl = kr_rank(K[u - 1]);
    if (kl != RANK_WALL) {
      if (kl < k) return false;
      const int lim = V.max_left[S[u]];
      int cum = L[u - 1] & LEN_MASK;
      for (int q = u - 2; q >= 0; --q) {
        const uint32_t kq = kr_rank(K[q]);
        if (kq == RANK_WALL) break;
        cum += L[q] & LEN_MASK;
        if (cum > lim) break;
        if (kq < k) return false;
      }
    }
  }
  if (i + 1 < m - 1) {
    const uint32_t kr = kr_rank(K[i + 1]);
    if (kr != RANK_WALL) {
      if (kr < k) return false;
      const int lim = V.max_right[S[i + 1]];
      int cum = L[i + 2] & LEN_MASK;
      for (int q = i + 2; q < m - 1; ++q) {
        const uint32_t kq = kr_rank(K[q]);
        if (kq == RANK_WALL) break;
        cum += L[q + 1] & LEN_MASK;
        if (cum > lim) break;
        if (kq < k) return false;
      }
    }
  }
  return true;
}

// block-wide scans for blockDim.x a multiple of 32; `sh` holds >= blockDim/32 words
__device__ __forceinline__ int block_excl_sum(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int k = 0; k < nw; ++k) {
    const int x = sh[k];
    pre += k < warp ? x : 0;
    tot += x;
  }
  *total = tot;
  __syncthreads();
  return pre + inc - v;
}

__device__ __forceinline__ int block_excl_max(int v, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc = max(inc, o);
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  int pre = -1;
  for (int k = 0; k < warp; ++k) pre = max(pre, sh[k]);
  const int ex = __shfl_up_sync(0xffffffffu, inc, 1);
  __syncthreads();
  return lane == 0 ? pre : max(pre, ex);
}

__device__ __forceinline__ unsigned long long block_min_u64(unsigned long long v, unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o < v ? o : v;
  }
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  unsigned long long r = ~0ull;
  for (int k = 0; k < nw; ++k) r = sh[k] < r ? sh[k] : r;
  __syncthreads();
  return r;
}

__device__ __forceinline__ bool bit_at(const uint32_t* bits, int p) { return (bits[p >> 5] >> (p & 31)) & 1u; }

// ---------------------------------------------------------------------------
// K3: the fragments that start in one 1 KiB chunk
//
// Most fragments need no merge loop: a single byte is its byte token, and a
// fragment whose bytes equal a token t with BPE(bytes(t)) == [t] (checked for
// every token at load time) encodes to [t].  One thread per fragment settles
// those with a hash probe; only the rest enter the sweep engine, in shared
// memory, with walls between fragments.

struct ChunkEngine {
  uint32_t sym[ENG_CAP];
  unsigned long long kr[ENG_CAP];
  uint16_t len[ENG_CAP];
  uint16_t rs[ENG_CAP];
  uint16_t fidx[ENG_CAP];      // fragment of each engine symbol
  uint8_t fl[ENG_CAP];
  uint8_t text[ENG_CAP];       // bytes [first, end)
  uint32_t bits[ENG_CAP / 32];
  uint16_t fstart[CHUNK + 1];  // fragment starts relative to `first`, then `end`
  int32_t ftok[CHUNK];         // settled token, or -1: goes through the engine
  int32_t fcnt[CHUNK];         // ids of each fragment
  uint16_t fout[CHUNK];        // first id of each fragment (relative)
  uint16_t feng[CHUNK];        // first engine symbol of each fragment
  int scan[ENG_THREADS / 32];
  unsigned long long scan64[ENG_THREADS / 32];
  int32_t byte_id[256];
  long long first, end, longfrag, item0;
  int nf;
};

__global__ void __launch_bounds__(ENG_THREADS) k_bpe_chunk(Call c, Workspace ws, DevVocab V) {
  extern __shared__ __align__(16) uint8_t dsm[];
  ChunkEngine& E = *reinterpret_cast<ChunkEngine*>(dsm);
  const int tid = threadIdx.x, T = ENG_THREADS;
  const long long chunk = blockIdx.x;
  const long long r0 = chunk * CHUNK;
  const long long r1 = min(r0 + CHUNK, c.n);
  const long long lim = min(r0 + ENG_CAP, c.n);
  E.byte_id[tid] = V.byte_id[tid];
  for (int w = tid; w < ENG_CAP / 32; w += T) {
    const long long p = r0 + 32ll * w;
    uint32_t v = 0;
    if (p < lim) {
      v = ws.pstart[(r0 >> 5) + w];
      if (lim - p < 32) v &= (1u << (lim - p)) - 1u;
    }
    E.bits[w] = v;
  }
  __syncthreads();
  if (tid < 32) {
    // first and last fragment start in [r0, r1); first start in [r1, lim)
    const int lane = tid;
    const uint32_t nz = __ballot_sync(0xffffffffu, E.bits[lane] != 0u);  // CHUNK / 32 == 32 words
    const uint32_t nz1 = __ballot_sync(0xffffffffu, E.bits[32 + lane] != 0u);
    if (lane == 0) {
      long long first = -1, last = -1, end = -1;
      if (nz) {
        const int a = __ffs(nz) - 1, b = 31 - __clz(nz);
        first = r0 + 32ll * a + (__ffs(E.bits[a]) - 1);
        last = r0 + 32ll * b + (31 - __clz(E.bits[b]));
      }
      if (r1 >= c.n) end = c.n;
      else if (nz1) { const int a = __ffs(nz1) - 1; end = r1 + 32ll * a + (__ffs(E.bits[32 + a]) - 1); }
      else if (lim >= c.n) end = c.n;
      long long lf = -1;
      if (first >= 0 && end < 0) {  // the last fragment runs past lim: queue it
        lf = last;
        end = last;
        const uint32_t q = atomicAdd(&ws.st->long_count, 1u);
        ws.longq[q] = Frag{last, chunk};
      }
      E.first = first;
      E.end = end;
      E.longfrag = lf;
    }
  }
  __syncthreads();
  const long long fs = E.first;
  if (fs < 0) {  // no fragment starts here (the chunk lies inside a long fragment)
    if (tid == 0) {
      ws.cm_first[chunk] = -1;
      ws.cm_count[chunk] = 0;
      ws.cm_long[chunk] = -1;
    }
    return;
  }
  const int span = (int)(E.end - fs);  // bytes of the fragments handled here
  const int rel = (int)(fs - r0);
  for (int i = tid; i < span; i += T) E.text[i] = c.text[fs + i];
  // fragment starts in [fs, min(r1, end)): thread t looks at 4 bit positions
  {
    const int q0 = tid * 4;  // positions relative to r0
    const uint32_t nib = (E.bits[q0 >> 5] >> (q0 & 31)) & 0xFu;
    uint32_t mine = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (((nib >> q) & 1u) && r0 + q0 + q < E.end) mine |= 1u << q;
    int nf = 0;
    int idx = block_excl_sum(__popc(mine), &nf, E.scan);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if ((mine >> q) & 1u) E.fstart[idx++] = (uint16_t)(q0 + q - rel);
    if (tid == 0) {
      E.nf = nf;
      E.fstart[nf] = (uint16_t)span;
    }
  }
  __syncthreads();
  const int nf = E.nf;
  // settle single bytes and whole tokens; contiguous fragments per thread
  const int FB = (nf + T - 1) / T;
  const int flo = min(tid * FB, nf), fhi = min(flo + FB, nf);
  int eng_bytes = 0;
  for (int f = flo; f < fhi; ++f) {
    const int a = E.fstart[f], L = E.fstart[f + 1] - a;
    int t = L == 1 ? E.byte_id[E.text[a]] : whole_lookup(V, E.text + a, L);
    E.ftok[f] = t;
    E.fcnt[f] = t >= 0 ? 1 : 0;
    if (t < 0) eng_bytes += L;
  }
  int m0 = 0;
  int eo = block_excl_sum(eng_bytes, &m0, E.scan);
  for (int f = flo; f < fhi; ++f) {
    if (E.ftok[f] >= 0) continue;
    const int a = E.fstart[f], L = E.fstart[f + 1] - a;
    for (int j = 0; j < L; ++j) {
      E.sym[eo + j] = (uint32_t)E.byte_id[E.text[a + j]];
      E.len[eo + j] = (uint16_t)(1u | (j == 0 ? FRAG_START : 0u));
      E.fidx[eo + j] = (uint16_t)f;
    }
    eo += L;
  }
  __syncthreads();
  for (int i = tid; i < m0; i += T)
    E.kr[i] = (i + 1 >= m0 || (E.len[i + 1] & FRAG_START)) ? KR_WALL : merge_lookup(V, E.sym[i], E.sym[i + 1]);
  __syncthreads();

  int m = m0;
  for (int sweep = 0; sweep <= m0; ++sweep) {
    const int B = (m + T - 1) / T;
    const int lo = min(tid * B, m), hi = min(lo + B, m);
    // A: any mergeable pair left?  run starts of equal-rank pairs
    bool anyk = false;
    int lastrun = -1;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = kr_rank(E.kr[i]);
      anyk |= mergeable(k);
      if (i == 0 || kr_rank(E.kr[i - 1]) != k) lastrun = i;
    }
    if (!__syncthreads_or(anyk)) break;
    int run = block_excl_max(lastrun, E.scan);
    for (int i = lo; i < hi; ++i) {
      if (i == 0 || kr_rank(E.kr[i - 1]) != kr_rank(E.kr[i])) run = i;
      E.rs[i] = (uint16_t)run;
    }
    __syncthreads();
    // B: safe pairs
    if (V.monotone) {
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(E.kr[i]);
        E.fl[i] = (mergeable(k) && pair_safe(V, E.sym, E.len, E.kr, E.rs, m, i, k)) ? 1 : 0;
      }
    } else {
      unsigned long long best = ~0ull;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(E.kr[i]);
        if (mergeable(k)) {
          const unsigned long long key = ((unsigned long long)k << 32) | (uint32_t)i;
          best = key < best ? key : best;
        }
      }
      best = block_min_u64(best, E.scan64);
      for (int i = lo; i < hi; ++i) E.fl[i] = ((uint32_t)best == (uint32_t)i) ? 1 : 0;
    }
    __syncthreads();
    // C: merge and compact, through registers
    uint32_t nsym[ENG_EPT];
    uint16_t nlen[ENG_EPT], nfi[ENG_EPT];
    unsigned long long nkr[ENG_EPT];
    uint32_t keep = 0;
#pragma unroll
    for (int j = 0; j < ENG_EPT; ++j) {
      const int i = lo + j;
      nsym[j] = 0; nlen[j] = 0; nkr[j] = 0; nfi[j] = 0;
      if (i < hi && !(i > 0 && E.fl[i - 1])) {
        keep |= 1u << j;
        const bool mg = E.fl[i] != 0;
        if (mg) {
          nsym[j] = kr_result(E.kr[i]);
          nlen[j] = (uint16_t)(((E.len[i] & LEN_MASK) + (E.len[i + 1] & LEN_MASK)) | (E.len[i] & FRAG_START));
        } else {
          nsym[j] = E.sym[i];
          nlen[j] = E.len[i];
        }
        nfi[j] = E.fidx[i];
        // an unchanged pair keeps its key; pairs touching a new symbol are looked up
        nkr[j] = (!mg && i + 1 < m && !E.fl[i + 1]) ? E.kr[i] : KR_NEED;
      }
    }
    int newm = 0;
    const int base = block_excl_sum(__popc(keep), &newm, E.scan);
#pragma unroll
    for (int j = 0; j < ENG_EPT; ++j) {
      if ((keep >> j) & 1u) {
        const int p = base + __popc(keep & ((1u << j) - 1u));
        E.sym[p] = nsym[j];
        E.len[p] = nlen[j];
        E.kr[p] = nkr[j];
        E.fidx[p] = nfi[j];
      }
    }
    __syncthreads();
    // D: keys of pairs that touch a new symbol
    const int cnt = __popc(keep);
    for (int p = base; p < base + cnt; ++p) {
      if (kr_rank(E.kr[p]) == RANK_NEED) {
        if (p + 1 >= newm || (E.len[p + 1] & FRAG_START)) E.kr[p] = KR_WALL;
        else E.kr[p] = merge_lookup(V, E.sym[p], E.sym[p + 1]);
      }
    }
    m = newm;
    __syncthreads();
    if (sweep == m0 && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);  // cannot happen: every sweep merges
  }
  // ids per fragment, then the fragments' first ids
  for (int i = tid; i < m; i += T) {
    const int f = E.fidx[i];
    if (E.len[i] & FRAG_START) E.feng[f] = (uint16_t)i;
    atomicAdd(&E.fcnt[f], 1);
  }
  __syncthreads();
  int ids = 0;
  for (int f = flo; f < fhi; ++f) ids += E.fcnt[f];
  int total = 0;
  int oo = block_excl_sum(ids, &total, E.scan);
  for (int f = flo; f < fhi; ++f) {
    E.fout[f] = (uint16_t)oo;
    oo += E.fcnt[f];
  }
  __syncthreads();
  for (int f = tid; f < nf; f += T)
    if (E.ftok[f] >= 0) ws.tok[fs + E.fout[f]] = E.ftok[f];
  for (int i = tid; i < m; i += T) {
    const int f = E.fidx[i];
    ws.tok[fs + E.fout[f] + (i - E.feng[f])] = (int32_t)E.sym[i];
  }
  if (tid == 0) {
    ws.cm_first[chunk] = fs;
    ws.cm_count[chunk] = total;
    ws.cm_long[chunk] = E.longfrag;
  }
  // batch: ids before each item start in this chunk (K5 adds the chunk's offset)
  if (c.item_off) {
    if (tid == 0) {
      int a = 0, b = c.n_items + 1;  // first item start >= r0
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (c.item[mid] < r0) a = mid + 1; else b = mid;
      }
      E.item0 = a;
    }
    __syncthreads();
    for (int k = (int)E.item0 + tid; k <= c.n_items; k += T) {
      const long long x = c.item[k];
      if (x >= r1) break;
      int a = 0, b = nf;  // fragment starting at x (or the long fragment after the last)
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (fs + E.fstart[mid] < x) a = mid + 1; else b = mid;
      }
      c.item_off[k] = a < nf ? E.fout[a] : total;
    }
  }
}

// ---------------------------------------------------------------------------
// K4: fragments longer than a chunk engine holds, one CTA each, in global
// memory at the fragment's byte offsets (double-buffered)

__global__ void __launch_bounds__(LONG_THREADS) k_bpe_long(Call c, Workspace ws, DevVocab V) {
  __shared__ int sh[LONG_THREADS / 32];
  __shared__ unsigned long long sh64[LONG_THREADS / 32];
  __shared__ uint32_t s_idx;
  __shared__ unsigned long long s_end;
  const int tid = threadIdx.x, T = blockDim.x;
  const uint32_t count = *(volatile uint32_t*)&ws.st->long_count;
  while (true) {
    if (tid == 0) s_idx = atomicAdd(&ws.st->long_taken, 1u);
    __syncthreads();
    const uint32_t idx = s_idx;
    __syncthreads();
    if (idx >= count) break;
    const Frag f = ws.longq[idx];
    // end: the next fragment start after f.start, or the text end
    if (tid == 0) s_end = (unsigned long long)c.n;
    __syncthreads();
    const long long w0 = (f.start + 1) >> 5, wn = (c.n + 31) >> 5;
    for (long long base = w0; base < wn; base += T) {
      const long long wi = base + tid;
      if (wi < wn) {
        uint32_t wv = ws.pstart[wi];
        if (wi == w0) wv &= ~0u << ((f.start + 1) & 31);
        if (wi * 32 + 32 > c.n) wv &= (c.n - wi * 32 >= 32) ? ~0u : ((1u << (c.n - wi * 32)) - 1u);
        if (wv) atomicMin(&s_end, (unsigned long long)(wi * 32 + __ffs(wv) - 1));
      }
      __syncthreads();
      const bool found = s_end < (unsigned long long)c.n;
      __syncthreads();
      if (found) break;
    }
    const long long a = f.start;
    const int m0 = (int)((long long)s_end - a);
    uint32_t* S0 = ws.e_sym[0] + a;
    uint32_t* S1 = ws.e_sym[1] + a;
    uint16_t* L0 = ws.e_len[0] + a;
    uint16_t* L1 = ws.e_len[1] + a;
    unsigned long long* K0 = ws.e_kr[0] + a;
    unsigned long long* K1 = ws.e_kr[1] + a;
    uint8_t* FL = ws.e_fl + a;
    int32_t* RS = ws.e_rs + a;
    for (int i = tid; i < m0; i += T) {
      S0[i] = (uint32_t)V.byte_id[c.text[a + i]];
      L0[i] = 1;
    }
    __syncthreads();
    for (int i = tid; i < m0; i += T) K0[i] = (i + 1 < m0) ? merge_lookup(V, S0[i], S0[i + 1]) : KR_WALL;
    __syncthreads();
    int m = m0, cur = 0;
    for (int sweep = 0; sweep <= m0; ++sweep) {
      uint32_t* S = cur ? S1 : S0;
      uint16_t* L = cur ? L1 : L0;
      unsigned long long* K = cur ? K1 : K0;
      uint32_t* S2 = cur ? S0 : S1;
      uint16_t* L2 = cur ? L0 : L1;
      unsigned long long* K2 = cur ? K0 : K1;
      const int B = (m + T - 1) / T;
      const int lo = min(tid * B, m), hi = min(lo + B, m);
      bool anyk = false;
      int lastrun = -1;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(K[i]);
        anyk |= mergeable(k);
        if (i == 0 || kr_rank(K[i - 1]) != k) lastrun = i;
      }
      if (!__syncthreads_or(anyk)) break;
      int run = block_excl_max(lastrun, sh);
      for (int i = lo; i < hi; ++i) {
        if (i == 0 || kr_rank(K[i - 1]) != kr_rank(K[i])) run = i;
        RS[i] = run;
      }
      __syncthreads();
      if (V.monotone) {
        for (int i = lo; i < hi; ++i) {
          const uint32_t k = kr_rank(K[i]);
          FL[i] = (mergeable(k) && pair_safe(V, S, L, K, RS, m, i, k)) ? 1 : 0;
        }
      } else {
        unsigned long long best = ~0ull;
        for (int i = lo; i < hi; ++i) {
          const uint32_t k = kr_rank(K[i]);
          if (mergeable(k)) {
            const unsigned long long key = ((unsigned long long)k << 32) | (uint32_t)i;
            best = key < best ? key : best;
          }
        }
        best = block_min_u64(best, sh64);
        for (int i = lo; i < hi; ++i) FL[i] = ((uint32_t)best == (uint32_t)i) ? 1 : 0;
      }
      __syncthreads();
      int keep = 0;
      for (int i = lo; i < hi; ++i) keep += !(i > 0 && FL[i - 1]);
      int newm = 0;
      int p = block_excl_sum(keep, &newm, sh);
      for (int i = lo; i < hi; ++i) {
        if (i > 0 && FL[i - 1]) continue;
        const bool mg = FL[i] != 0;
        S2[p] = mg ? kr_result(K[i]) : S[i];
        L2[p] = mg ? (uint16_t)(L[i] + L[i + 1]) : L[i];
        K2[p] = (!mg && i + 1 < m && !FL[i + 1]) ? K[i] : KR_NEED;
        ++p;
      }
      __syncthreads();
      for (int q = tid; q < newm; q += T) {
        if (kr_rank(K2[q]) == RANK_NEED) K2[q] = (q + 1 >= newm) ? KR_WALL : merge_lookup(V, S2[q], S2[q + 1]);
      }
      __syncthreads();
      cur ^= 1;
      m = newm;
      if (sweep == m0 && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);
    }
    const uint32_t* S = cur ? S1 : S0;
    for (int i = tid; i < m; i += T) ws.tok[a + i] = (int32_t)S[i];
    if (tid == 0) ws.cm_long_count[f.chunk] = m;
    __syncthreads();
  }
}

void launch_bpe_chunk(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaFuncSetAttribute(k_bpe_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(ChunkEngine));
    attr_set[dev] = true;
  }
  k_bpe_chunk<<<(unsigned)n_chunks(c.n), ENG_THREADS, sizeof(ChunkEngine), s>>>(c, w, v);
}

void launch_bpe_long(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_long<<<n_sms, LONG_THREADS, 0, s>>>(c, w, v);
}

}  // namespace tokgb
