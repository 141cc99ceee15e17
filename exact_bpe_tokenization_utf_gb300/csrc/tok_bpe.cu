// Per-fragment BPE, E ("TokTier: exact stateful tokenization for agentic LLM
// serving", Section 4.2): every fragment is encoded on its own by merging the
// lowest-rank adjacent pair (leftmost on ties) until no adjacent pair is a
// merge.  The pages tier fragments by length (one thread, one warp, one block
// per fragment); here one CTA encodes all fragments of a 512-byte chunk at
// once, and only fragments longer than 512 bytes get a CTA each.
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

// Is pair i (rank k) safe to merge now?  u is the first pair of the run of
// equal-rank pairs that contains i; ml(x) / mr(x) are the longest left /
// right operand of any merge whose right / left operand is symbol x.  See the
// file comment.
template <class ML, class MR>
__device__ __forceinline__ bool pair_safe(const uint16_t* L, const unsigned long long* K, int m, int i, int u,
                                          uint32_t k, ML ml, MR mr) {
  if ((i - u) & 1) return false;
  if (u > 0) {
    const uint32_t kl = kr_rank(K[u - 1]);
    if (kl != RANK_WALL) {
      if (kl < k) return false;
      const int lim = ml(u);
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
      const int lim = mr(i + 1);
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
// K3: the fragments that start in one 512-byte chunk
//
// Most fragments need no merge loop: a single byte is its byte token, and a
// fragment whose bytes equal a token t with BPE(bytes(t)) == [t] (checked for
// every token at load time) encodes to [t].  One thread per fragment settles
// those with a hash probe; the rest go through the sweep engine in shared
// memory, in batches of at most B_CAP symbols, with walls between fragments.
// Each symbol carries its operand-length bounds, so the safety test reads
// shared memory only; the merge lookups of a sweep are issued before its
// compaction scan.

struct ChunkEngine {
  // one engine batch
  uint32_t sym[B_CAP];
  unsigned long long kr[B_CAP];
  uint16_t len[B_CAP];      // byte length | FRAG_START
  uint16_t rs[B_CAP];       // run start of equal-rank pairs
  uint16_t fidx[B_CAP];     // fragment of each symbol
  uint16_t ml[B_CAP];       // longest left operand of merges whose right operand is this symbol
  uint16_t mr[B_CAP];       // longest right operand of merges whose left operand is this symbol
  uint8_t fl[B_CAP];        // pair merges this sweep
  // the CTA's bytes and fragment starts
  uint8_t text[B_RANGE];
  uint32_t bits[B_RANGE / 32];
  // fragments that start in the chunk (at most BCHUNK)
  uint16_t fstart[BCHUNK + 1];  // relative to `first`; then the span
  int32_t ftok[BCHUNK];         // settled token, or -1
  int32_t fcnt[BCHUNK];         // ids of each fragment
  uint16_t fout[BCHUNK];        // first id of each fragment
  uint16_t feng[BCHUNK];        // first engine symbol of a fragment in its batch
  uint16_t feoff[BCHUNK];       // offset of an unresolved fragment among all unresolved bytes
  uint16_t ulist[BCHUNK];       // unresolved fragments in order
  uint16_t ueoff[BCHUNK + 1];   // their offsets, then the total
  uint32_t efinal[B_RANGE];     // engine results at their fragment's feoff
  int32_t byte_id[256];
  uint16_t byte_ml[256], byte_mr[256];
  int scan[B_THREADS / 32];
  unsigned long long scan64[B_THREADS / 32];
  long long first, end, longfrag, item0;
  int nf, nu, sflags, batch_end;
};

__global__ void __launch_bounds__(B_THREADS) k_bpe_chunk(Call c, Workspace ws, DevVocab V) {
  extern __shared__ __align__(16) uint8_t dsm[];
  ChunkEngine& E = *reinterpret_cast<ChunkEngine*>(dsm);
  const int tid = threadIdx.x, T = B_THREADS, lane = tid & 31;
  const long long chunk = blockIdx.x;
  const long long r0 = chunk * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  const long long lim = min(r0 + B_RANGE, c.n);
  for (int b = tid; b < 256; b += T) {
    const int32_t id = V.byte_id[b];
    E.byte_id[b] = id;
    E.byte_ml[b] = V.max_left[id];
    E.byte_mr[b] = V.max_right[id];
  }
  if (tid < B_RANGE / 32) {
    const long long p = r0 + 32ll * tid;
    uint32_t v = 0;
    if (p < lim) {
      v = ws.pstart[(r0 >> 5) + tid];
      if (lim - p < 32) v &= (1u << (lim - p)) - 1u;
    }
    E.bits[tid] = v;
  }
  if (tid == 0) E.sflags = 0;
  __syncthreads();
  if (tid < 32) {
    // first and last fragment start in [r0, r1) (words 0..15), first start in [r1, lim) (16..31)
    const uint32_t w = E.bits[lane];
    const uint32_t nz = __ballot_sync(0xffffffffu, lane < BCHUNK / 32 && w != 0u);
    const uint32_t nz1 = __ballot_sync(0xffffffffu, lane >= BCHUNK / 32 && w != 0u) >> (BCHUNK / 32);
    if (lane == 0) {
      long long first = -1, last = -1, end = -1;
      if (nz) {
        const int a = __ffs(nz) - 1, b = 31 - __clz(nz);
        first = r0 + 32ll * a + (__ffs(E.bits[a]) - 1);
        last = r0 + 32ll * b + (31 - __clz(E.bits[b]));
      }
      if (r1 >= c.n) end = c.n;
      else if (nz1) {
        const int a = __ffs(nz1) - 1;
        end = r1 + 32ll * a + (__ffs(E.bits[BCHUNK / 32 + a]) - 1);
      } else if (lim >= c.n) end = c.n;
      long long lf = -1;
      if (first >= 0 && (end < 0 || end - last > B_CAP)) {  // the last fragment is long: queue it
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
  const int span = (int)(E.end - fs);
  const int rel = (int)(fs - r0);
  for (int i = tid; i < span; i += T) E.text[i] = c.text[fs + i];
  {  // fragment starts in [fs, min(r1, end)): thread t looks at 4 bit positions
    const int q0 = tid * 4;
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
  // settle single bytes and whole tokens (contiguous fragments per thread)
  const int FB = (nf + T - 1) / T;
  const int flo = min(tid * FB, nf), fhi = min(flo + FB, nf);
  int ubytes = 0, ucount = 0;
  for (int f = flo; f < fhi; ++f) {
    const int a = E.fstart[f], L = E.fstart[f + 1] - a;
    const int t = L == 1 ? E.byte_id[E.text[a]] : whole_lookup(V, E.text + a, L);
    E.ftok[f] = t;
    E.fcnt[f] = t >= 0 ? 1 : 0;
    if (t < 0) { ubytes += L; ++ucount; }
  }
  int nu = 0, ub_all = 0;
  int ui = block_excl_sum(ucount, &nu, E.scan);
  int uo = block_excl_sum(ubytes, &ub_all, E.scan);
  for (int f = flo; f < fhi; ++f) {
    if (E.ftok[f] >= 0) continue;
    E.ulist[ui] = (uint16_t)f;
    E.ueoff[ui] = (uint16_t)uo;
    E.feoff[f] = (uint16_t)uo;
    ++ui;
    uo += E.fstart[f + 1] - E.fstart[f];
  }
  if (tid == 0) E.ueoff[nu] = (uint16_t)ub_all;
  __syncthreads();

  // engine batches over the unresolved fragments
  for (int ub = 0; ub < nu;) {
    if (tid == 0) {  // largest ue with ueoff[ue] - ueoff[ub] <= B_CAP
      int a = ub + 1, b = nu;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (E.ueoff[mid] - E.ueoff[ub] <= B_CAP) a = mid; else b = mid - 1;
      }
      E.batch_end = a;
    }
    __syncthreads();
    const int ue = E.batch_end;
    const int base = E.ueoff[ub];
    const int M = E.ueoff[ue] - base;
    for (int i = tid; i < M; i += T) {
      int a = ub, b = ue - 1;  // fragment k with ueoff[k] <= base + i < ueoff[k+1]
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (E.ueoff[mid] <= base + i) a = mid; else b = mid - 1;
      }
      const int f = E.ulist[a];
      const int j = base + i - E.ueoff[a];
      const uint8_t byte = E.text[E.fstart[f] + j];
      E.sym[i] = (uint32_t)E.byte_id[byte];
      E.len[i] = (uint16_t)(1u | (j == 0 ? FRAG_START : 0u));
      E.fidx[i] = (uint16_t)f;
      E.ml[i] = E.byte_ml[byte];
      E.mr[i] = E.byte_mr[byte];
    }
    __syncthreads();
    for (int i = tid; i < M; i += T)
      E.kr[i] = (i + 1 >= M || (E.len[i + 1] & FRAG_START)) ? KR_WALL : merge_lookup(V, E.sym[i], E.sym[i + 1]);
    __syncthreads();

    int m = M;
    for (int sweep = 0; sweep <= M; ++sweep) {
      const int B = (m + T - 1) / T;
      const int lo = min(tid * B, m), hi = min(lo + B, m);
      // A: any mergeable pair left?  any overlapping equal-rank pairs?
      int fl2 = 0;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(E.kr[i]);
        if (mergeable(k)) {
          fl2 |= 1;
          if (i > 0 && kr_rank(E.kr[i - 1]) == k) fl2 |= 2;
        }
      }
      fl2 = __reduce_or_sync(0xffffffffu, fl2);
      if (lane == 0 && fl2) atomicOr(&E.sflags, fl2);
      __syncthreads();
      const int flags = E.sflags;
      if (!(flags & 1)) break;
      if (flags & 2) {
        int lastrun = -1;
        for (int i = lo; i < hi; ++i)
          if (i == 0 || kr_rank(E.kr[i - 1]) != kr_rank(E.kr[i])) lastrun = i;
        int run = block_excl_max(lastrun, E.scan);
        for (int i = lo; i < hi; ++i) {
          if (i == 0 || kr_rank(E.kr[i - 1]) != kr_rank(E.kr[i])) run = i;
          E.rs[i] = (uint16_t)run;
        }
        __syncthreads();
      }
      // B: safe pairs
      if (V.monotone) {
        auto mlf = [&](int x) { return (int)E.ml[x]; };
        auto mrf = [&](int x) { return (int)E.mr[x]; };
        for (int i = lo; i < hi; ++i) {
          const uint32_t k = kr_rank(E.kr[i]);
          const int u = (flags & 2) ? (int)E.rs[i] : i;
          E.fl[i] = (mergeable(k) && pair_safe(E.len, E.kr, m, i, u, k, mlf, mrf)) ? 1 : 0;
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
      // C: merge, look up the new pairs, compact
      uint32_t nsym[B_EPT];
      uint16_t nlen[B_EPT], nfi[B_EPT], nml[B_EPT], nmr[B_EPT];
      unsigned long long nkr[B_EPT];
      uint32_t keep = 0;
#pragma unroll
      for (int j = 0; j < B_EPT; ++j) {
        const int i = lo + j;
        nsym[j] = 0; nlen[j] = 0; nfi[j] = 0; nml[j] = 0; nmr[j] = 0; nkr[j] = KR_WALL;
        if (i < hi && !(i > 0 && E.fl[i - 1])) {
          keep |= 1u << j;
          const bool mg = E.fl[i] != 0;
          if (mg) {
            const uint32_t r = kr_result(E.kr[i]);
            nsym[j] = r;
            nlen[j] = (uint16_t)(((E.len[i] & LEN_MASK) + (E.len[i + 1] & LEN_MASK)) | (E.len[i] & FRAG_START));
            nml[j] = __ldg(V.max_left + r);
            nmr[j] = __ldg(V.max_right + r);
          } else {
            nsym[j] = E.sym[i];
            nlen[j] = E.len[i];
            nml[j] = E.ml[i];
            nmr[j] = E.mr[i];
          }
          nfi[j] = E.fidx[i];
          const int jn = mg ? i + 2 : i + 1;  // the next symbol that survives
          if (jn >= m || (E.len[jn] & FRAG_START)) nkr[j] = KR_WALL;
          else if (!mg && !E.fl[jn]) nkr[j] = E.kr[i];  // unchanged pair keeps its key
          else nkr[j] = merge_lookup(V, nsym[j], E.fl[jn] ? kr_result(E.kr[jn]) : E.sym[jn]);
        }
      }
      int newm = 0;
      const int bpos = block_excl_sum(__popc(keep), &newm, E.scan);
#pragma unroll
      for (int j = 0; j < B_EPT; ++j) {
        if ((keep >> j) & 1u) {
          const int p = bpos + __popc(keep & ((1u << j) - 1u));
          E.sym[p] = nsym[j];
          E.len[p] = nlen[j];
          E.kr[p] = nkr[j];
          E.fidx[p] = nfi[j];
          E.ml[p] = nml[j];
          E.mr[p] = nmr[j];
        }
      }
      if (tid == 0) E.sflags = 0;
      m = newm;
      __syncthreads();
      if (sweep == M && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);  // cannot happen: every sweep merges
    }
    // this batch's results
    for (int i = tid; i < m; i += T) {
      const int f = E.fidx[i];
      if (E.len[i] & FRAG_START) E.feng[f] = (uint16_t)i;
      atomicAdd(&E.fcnt[f], 1);
    }
    __syncthreads();
    for (int i = tid; i < m; i += T) {
      const int f = E.fidx[i];
      E.efinal[E.feoff[f] + (i - E.feng[f])] = E.sym[i];
    }
    if (tid == 0) E.sflags = 0;
    __syncthreads();
    ub = ue;
  }
  // first id of each fragment, then the ids
  int ids = 0;
  for (int f = flo; f < fhi; ++f) ids += E.fcnt[f];
  int total = 0;
  int oo = block_excl_sum(ids, &total, E.scan);
  for (int f = flo; f < fhi; ++f) {
    E.fout[f] = (uint16_t)oo;
    oo += E.fcnt[f];
  }
  __syncthreads();
  for (int f = tid; f < nf; f += T) {
    const int o = E.fout[f];
    if (E.ftok[f] >= 0) {
      ws.tok[fs + o] = E.ftok[f];
    } else {
      const int e0 = E.feoff[f], cnt = E.fcnt[f];
      for (int j = 0; j < cnt; ++j) ws.tok[fs + o + j] = (int32_t)E.efinal[e0 + j];
    }
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
          FL[i] = (mergeable(k) && pair_safe(L, K, m, i, RS[i], k, [&](int x) { return (int)V.max_left[S[x]]; },
                                             [&](int x) { return (int)V.max_right[S[x]]; }))
                      ? 1
                      : 0;
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
  k_bpe_chunk<<<(unsigned)n_bchunks(c.n), B_THREADS, sizeof(ChunkEngine), s>>>(c, w, v);
}

void launch_bpe_long(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_long<<<n_sms, LONG_THREADS, 0, s>>>(c, w, v);
}

}  // namespace tokgb
