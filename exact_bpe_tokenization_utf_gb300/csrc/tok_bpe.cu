// Per-fragment BPE, E ("TokTier: exact stateful tokenization for agentic LLM
// serving", Section 4.2): every fragment is encoded on its own by merging the
// lowest-rank adjacent pair (leftmost on ties) until no adjacent pair is a
// merge.  The pages tier fragments by length (one thread, one warp, one block
// per fragment).  Here most fragments are settled by one probe (single bytes,
// whole self-encoding tokens); of the rest, those of at most 32 bytes share a
// warp, one symbol per lane, several fragments per warp (merged step by step
// when all are at most 16 bytes, else in sweeps); fragments of 33..B_CAP
// bytes get a CTA with shared memory, longer ones a CTA with global memory.
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

__device__ __forceinline__ unsigned long long block_excl_sum64(unsigned long long v, unsigned long long* total,
                                                               unsigned long long* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  unsigned long long pre = 0, tot = 0;
  for (int k = 0; k < nw; ++k) {
    const unsigned long long x = sh[k];
    pre += k < warp ? x : 0ull;
    tot += x;
  }
  *total = tot;
  __syncthreads();
  return pre + inc - v;
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
// Fragment engine over global memory: one fragment of m0 bytes at byte
// offset a, all threads of the CTA, arrays double-buffered at the fragment's
// byte offsets.  The same sweep as the shared-memory engine.  Writes the ids
// to out[0..m) and returns m (the same value in every thread).

__device__ int global_engine(const Call& c, const Workspace& ws, const DevVocab& V, long long a, int m0,
                             int32_t* out, int* sh, unsigned long long* sh64) {
  const int tid = threadIdx.x, T = blockDim.x;
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
    if (sweep == m0 && tid == 0) set_error(ws.st, ST_EINTERNAL);
  }
  const uint32_t* S = cur ? S1 : S0;
  for (int i = tid; i < m; i += T) out[i] = (int32_t)S[i];
  __syncthreads();
  return m;
}

// ---------------------------------------------------------------------------
// Engine storage

struct WarpBuf {            // one warp's compaction buffer, and the pair ranks for window walks
  uint32_t sym[32];
  unsigned long long kr[32];
  uint16_t len[32];         // byte length | FRAG_START
  uint16_t fidx[32];
  uint16_t ml[32];
  uint16_t mr[32];
  uint32_t rank[32];        // rank of pair (i, i+1) this sweep
  uint16_t blen[32];        // byte length of symbol i this sweep
};

struct CtaBatch {           // one batch of the CTA engine
  uint32_t sym[B_CAP];
  unsigned long long kr[B_CAP];
  uint16_t len[B_CAP];      // byte length | FRAG_START
  uint16_t rs[B_CAP];       // run start of equal-rank pairs
  uint16_t fidx[B_CAP];     // fragment of each symbol
  uint16_t ml[B_CAP];       // longest left operand of merges whose right operand is this symbol
  uint16_t mr[B_CAP];       // longest right operand of merges whose left operand is this symbol
  uint8_t fl[B_CAP];        // pair merges this sweep
};

// ---------------------------------------------------------------------------
// K3b: queued fragments of at most B_CAP bytes
//
// A persistent grid.  First every CTA takes fragments of 33..B_CAP bytes one
// at a time through the shared-memory engine; then every warp takes batches
// of short fragments through the warp engine.  Both write a fragment's ids at
// its byte offset in `tok` and their number at the same offset in `fcnt`.

// One fragment of M (33..B_CAP) bytes at byte offset a, all threads of the CTA.
__device__ void cta_fragment(const Call& c, const Workspace& ws, const DevVocab& V, long long a, int M, CtaBatch& C,
                             int* scan, unsigned long long* scan64, int* sflags) {
  const int tid = threadIdx.x, T = B_THREADS, lane = tid & 31;
  for (int i = tid; i < M; i += T) {
    const int32_t id = __ldg(V.byte_id + c.text[a + i]);
    C.sym[i] = (uint32_t)id;
    C.len[i] = (uint16_t)(1u | (i == 0 ? FRAG_START : 0u));
    C.ml[i] = __ldg(V.max_left + id);
    C.mr[i] = __ldg(V.max_right + id);
  }
  if (tid == 0) *sflags = 0;
  __syncthreads();
  // a byte pair that no merge result holds is a wall from the start: no
  // merge ever crosses it, so the pieces between walls encode apart (fewer
  // sweeps: the safe-pair walks stop at walls)
  for (int i = tid; i < M; i += T) {
    bool wall = i + 1 >= M;
    if (!wall && V.pair_bits) wall = !bit_at(V.pair_bits, ((int)c.text[a + i] << 8) | (int)c.text[a + i + 1]);
    C.kr[i] = wall ? KR_WALL : merge_lookup(V, C.sym[i], C.sym[i + 1]);
  }
  __syncthreads();
  int m = M;
  for (int sweep = 0; sweep <= M; ++sweep) {
    const int B = (m + T - 1) / T;
    const int lo = min(tid * B, m), hi = min(lo + B, m);
    // A: any mergeable pair left?  any overlapping equal-rank pairs?
    int fl2 = 0;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = kr_rank(C.kr[i]);
      if (mergeable(k)) {
        fl2 |= 1;
        if (i > 0 && kr_rank(C.kr[i - 1]) == k) fl2 |= 2;
      }
    }
    fl2 = __reduce_or_sync(0xffffffffu, fl2);
    if (lane == 0 && fl2) atomicOr(sflags, fl2);
    __syncthreads();
    const int flags = *sflags;
    if (!(flags & 1)) break;
    if (flags & 2) {
      int lastrun = -1;
      for (int i = lo; i < hi; ++i)
        if (i == 0 || kr_rank(C.kr[i - 1]) != kr_rank(C.kr[i])) lastrun = i;
      int run = block_excl_max(lastrun, scan);
      for (int i = lo; i < hi; ++i) {
        if (i == 0 || kr_rank(C.kr[i - 1]) != kr_rank(C.kr[i])) run = i;
        C.rs[i] = (uint16_t)run;
      }
      __syncthreads();
    }
    // B: safe pairs
    if (V.monotone) {
      auto mlf = [&](int x) { return (int)C.ml[x]; };
      auto mrf = [&](int x) { return (int)C.mr[x]; };
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(C.kr[i]);
        const int u = (flags & 2) ? (int)C.rs[i] : i;
        C.fl[i] = (mergeable(k) && pair_safe(C.len, C.kr, m, i, u, k, mlf, mrf)) ? 1 : 0;
      }
    } else {
      unsigned long long best = ~0ull;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(C.kr[i]);
        if (mergeable(k)) {
          const unsigned long long key = ((unsigned long long)k << 32) | (uint32_t)i;
          best = key < best ? key : best;
        }
      }
      best = block_min_u64(best, scan64);
      for (int i = lo; i < hi; ++i) C.fl[i] = ((uint32_t)best == (uint32_t)i) ? 1 : 0;
    }
    __syncthreads();
    // C: merge, look up the new pairs, compact
    uint32_t nsym[B_EPT];
    uint16_t nlen[B_EPT], nml[B_EPT], nmr[B_EPT];
    unsigned long long nkr[B_EPT];
    uint32_t keep = 0;
#pragma unroll
    for (int j = 0; j < B_EPT; ++j) {
      const int i = lo + j;
      nsym[j] = 0; nlen[j] = 0; nml[j] = 0; nmr[j] = 0; nkr[j] = KR_WALL;
      if (i < hi && !(i > 0 && C.fl[i - 1])) {
        keep |= 1u << j;
        const bool mg = C.fl[i] != 0;
        if (mg) {
          const uint32_t r = kr_result(C.kr[i]);
          nsym[j] = r;
          nlen[j] = (uint16_t)(((C.len[i] & LEN_MASK) + (C.len[i + 1] & LEN_MASK)) | (C.len[i] & FRAG_START));
          nml[j] = __ldg(V.max_left + r);
          nmr[j] = __ldg(V.max_right + r);
        } else {
          nsym[j] = C.sym[i];
          nlen[j] = C.len[i];
          nml[j] = C.ml[i];
          nmr[j] = C.mr[i];
        }
        const int jn = mg ? i + 2 : i + 1;  // the next symbol that survives
        // a wall before it stays (no merge crosses a wall)
        if (jn >= m || kr_rank(mg ? C.kr[i + 1] : C.kr[i]) == RANK_WALL) nkr[j] = KR_WALL;
        else if (!mg && !C.fl[jn]) nkr[j] = C.kr[i];  // unchanged pair keeps its key
        else nkr[j] = merge_lookup(V, nsym[j], C.fl[jn] ? kr_result(C.kr[jn]) : C.sym[jn]);
      }
    }
    int newm = 0;
    const int bpos = block_excl_sum(__popc(keep), &newm, scan);
#pragma unroll
    for (int j = 0; j < B_EPT; ++j) {
      if ((keep >> j) & 1u) {
        const int p = bpos + __popc(keep & ((1u << j) - 1u));
        C.sym[p] = nsym[j];
        C.len[p] = nlen[j];
        C.kr[p] = nkr[j];
        C.ml[p] = nml[j];
        C.mr[p] = nmr[j];
      }
    }
    if (tid == 0) *sflags = 0;
    m = newm;
    __syncthreads();
    if (sweep == M && tid == 0) set_error(ws.st, ST_EINTERNAL);  // cannot happen: every sweep merges
  }
  for (int i = tid; i < m; i += T) ws.tok[a + i] = (int32_t)C.sym[i];
  if (tid == 0) {
    ws.fcnt[a] = m;
    atomicAdd(&ws.ctot[a / BCHUNK], (uint32_t)m);
    atomicAdd(&ws.gtot[a / BCHUNK / CTOT_GROUP], (uint32_t)m);
  }
  __syncthreads();
}

// Sweep engine of one warp over a batch of M <= 32 symbols (lane i holds
// symbol i; lanes >= M are empty).  sym / lenb / fst / fid / mlv / mrv / kr
// are the lane's symbol, byte length, fragment-start flag, fragment, operand
// bounds and the key of pair (i, i+1) (KR_WALL across fragments and past the
// last symbol).  On return lane i < m holds the i-th result symbol.
__device__ __forceinline__ int warp_sweeps(WarpBuf& B, const DevVocab& V, DevStatus* st, int m, uint32_t& sym,
                                           uint32_t& lenb, bool& fst, int& fid, uint32_t& mlv, uint32_t& mrv,
                                           unsigned long long& kr) {
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  for (int sweep = 0; sweep <= 32; ++sweep) {
    const uint32_t k = kr_rank(kr);
    const bool mrg = mergeable(k);
    if (!__any_sync(FULL, mrg)) break;
    if (sweep == 32) {  // cannot happen: every sweep merges at least one pair
      if (lane == 0) set_error(st, ST_EINTERNAL);
      break;
    }
    uint32_t kl = __shfl_up_sync(FULL, k, 1);
    if (lane == 0) kl = RANK_WALL;
    uint32_t kn = __shfl_down_sync(FULL, k, 1);
    if (lane == 31) kn = RANK_WALL;
    // start u of the run of equal-rank pairs that contains pair i
    int u = lane;
    if (__any_sync(FULL, mrg && kl == k)) {
      int s = (mrg && kl != k) ? lane : -1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(FULL, s, off);
        if (lane >= off) s = max(s, o);
      }
      if (mrg && s >= 0) u = s;
    }
    bool safe = false;
    if (V.monotone) {
      // lowest rank over the fragment's pairs up to this one (pm) and from
      // this one on (sm); a wall pair is a segment of its own with no rank
      const bool wall = k == RANK_WALL;
      const uint32_t v = mrg ? k : NO_RANK;
      uint32_t pm = v, sm = v;
      bool pf = lane == 0 || wall || kl == RANK_WALL;
      bool ef = lane == 31 || wall || kn == RANK_WALL;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o1 = __shfl_up_sync(FULL, pm, off);
        const bool f1 = __shfl_up_sync(FULL, pf, off);
        const uint32_t o2 = __shfl_down_sync(FULL, sm, off);
        const bool f2 = __shfl_down_sync(FULL, ef, off);
        if (lane >= off) {
          if (!pf) pm = min(pm, o1);
          pf = pf || f1;
        }
        if (lane + off < 32) {
          if (!ef) sm = min(sm, o2);
          ef = ef || f2;
        }
      }
      const uint32_t pm_u2 = __shfl_sync(FULL, pm, max(u - 2, 0));
      const uint32_t kl_u = __shfl_sync(FULL, k, max(u - 1, 0));
      const uint32_t sm_i2 = __shfl_sync(FULL, sm, min(lane + 2, 31));
      const uint32_t ml_u = __shfl_sync(FULL, mlv, u);
      const uint32_t mr_i1 = __shfl_sync(FULL, mrv, min(lane + 1, 31));
      const bool has_l = u > 0 && kl_u != RANK_WALL;  // pair u-1 lies in the fragment
      const bool has_r = kn != RANK_WALL;             // pair i+1 lies in the fragment
      bool need = false;
      if (mrg) {
        const bool nbr_ok = ((lane - u) & 1) == 0 && (!has_l || kl_u >= k) && kn >= k;
        const bool left_clear = !has_l || u < 2 || pm_u2 >= k;
        const bool right_clear = !has_r || sm_i2 >= k;
        safe = nbr_ok && left_clear && right_clear;
        need = nbr_ok && !(left_clear && right_clear);
      }
      // a lower rank further away: walk the length-bounded windows, each lane
      // on its own through the ranks and lengths in shared memory
      if (__any_sync(FULL, need)) {
        B.rank[lane] = k;
        B.blen[lane] = (uint16_t)lenb;
        __syncwarp();
        if (need) {
          bool ok = true;
          if (has_l && u >= 2) {
            // left: a token grown from pair q <= u-2 ends at symbol u-1
            int cum = B.blen[u - 1];
            for (int q = u - 2; q >= 0; --q) {
              const uint32_t kq = B.rank[q];
              if (kq == RANK_WALL) break;
              cum += B.blen[q];
              if (cum > (int)ml_u) break;
              if (kq < k) { ok = false; break; }
            }
          }
          if (ok && has_r) {
            // right: a token grown from pair q >= i+2 starts at symbol i+2
            int cum = lane + 2 < 32 ? B.blen[lane + 2] : 0;
            for (int q = lane + 2; q < 31; ++q) {
              const uint32_t kq = B.rank[q];
              if (kq == RANK_WALL) break;
              cum += B.blen[q + 1];
              if (cum > (int)mr_i1) break;
              if (kq < k) { ok = false; break; }
            }
          }
          safe = ok;
        }
        __syncwarp();
      }
    } else {
      // the rule itself: the leftmost lowest-rank pair of the batch
      unsigned long long best = mrg ? (((unsigned long long)k << 5) | (unsigned)lane) : ~0ull;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(FULL, best, off);
        best = o < best ? o : best;
      }
      safe = mrg && best != ~0ull && (int)(best & 31u) == lane;
    }
    // merge: a safe pair's left symbol takes the result, its right one goes
    const bool absorbed = __shfl_up_sync(FULL, safe, 1) && lane > 0;
    const uint32_t res = kr_result(kr);
    const uint32_t nsym = safe ? res : sym;
    const uint32_t lnext = __shfl_down_sync(FULL, lenb, 1);
    const uint32_t nlen = safe ? lenb + lnext : lenb;
    uint32_t nml = mlv, nmr = mrv;
    if (safe) {
      nml = __ldg(V.max_left + res);
      nmr = __ldg(V.max_right + res);
    }
    // the next surviving symbol j = i+1, or i+2 after a merge
    const bool safe1 = __shfl_down_sync(FULL, safe, 1);
    const bool safe2 = __shfl_down_sync(FULL, safe, 2);
    const uint32_t sym1 = __shfl_down_sync(FULL, sym, 1);
    const uint32_t sym2 = __shfl_down_sync(FULL, sym, 2);
    const uint32_t res1 = __shfl_down_sync(FULL, res, 1);
    const uint32_t res2 = __shfl_down_sync(FULL, res, 2);
    const bool fs1 = __shfl_down_sync(FULL, fst, 1);
    const bool fs2 = __shfl_down_sync(FULL, fst, 2);
    const bool keep = lane < m && !absorbed;
    const int j = safe ? lane + 2 : lane + 1;
    const bool jfs = safe ? fs2 : fs1;
    const bool jsafe = safe ? safe2 : safe1;
    const uint32_t jsym = safe ? (safe2 ? res2 : sym2) : (safe1 ? res1 : sym1);
    unsigned long long nkr = KR_WALL;
    if (keep && j < m && !jfs) nkr = (!safe && !jsafe) ? kr : merge_lookup(V, nsym, jsym);
    // compaction through the warp's buffer
    const uint32_t kmask = __ballot_sync(FULL, keep);
    if (keep) {
      const int p = __popc(kmask & ((1u << lane) - 1u));
      B.sym[p] = nsym;
      B.len[p] = (uint16_t)(nlen | (fst ? FRAG_START : 0u));
      B.kr[p] = nkr;
      B.fidx[p] = (uint16_t)fid;
      B.ml[p] = (uint16_t)nml;
      B.mr[p] = (uint16_t)nmr;
    }
    __syncwarp();
    m = __popc(kmask);
    if (lane < m) {
      sym = B.sym[lane];
      const uint32_t l = B.len[lane];
      lenb = l & LEN_MASK;
      fst = (l & FRAG_START) != 0;
      kr = B.kr[lane];
      fid = B.fidx[lane];
      mlv = B.ml[lane];
      mrv = B.mr[lane];
    } else {
      sym = 0; lenb = 0; fst = false; kr = KR_WALL; fid = 0; mlv = 0; mrv = 0;
    }
    __syncwarp();
  }
  return m;
}


// Step engine of one warp over a batch of m <= 32 symbols (lane i holds
// symbol i; lanes >= m are empty): every step, each fragment of the batch
// merges its leftmost lowest-rank pair -- the rule itself, one merge at a
// time per fragment, for any vocabulary.  A step is a minimum of
// rank << 5 | lane over each fragment's lanes (one warp reduction with the
// fragment's lanes as the member mask, every fragment at once), the merge,
// one lookup per lane at most (the new symbol with its right neighbour, its
// left neighbour with it) and a compaction.  sym / lenb / fst / fid / kr are the lane's symbol, byte
// length, fragment-start flag, fragment and the key of pair (i, i+1)
// (KR_WALL across fragments and past the last symbol).  Ranks are below
// 2^20 (fewer merges than tokens), so rank << 5 | lane fits in 31 bits.
constexpr int STEP_MAX_LEN = 16;  // longest fragment of a batch for the step engine
constexpr uint32_t SEG_VAL = 0x7FFFFFFFu;  // no mergeable pair

__device__ __forceinline__ int warp_steps(WarpBuf& B, const DevVocab& V, DevStatus* st, int m, uint32_t& sym,
                                          uint32_t& lenb, bool& fst, int& fid, unsigned long long& kr) {
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  // Symbols stay in their lanes: a merge keeps the left lane and retires the
  // right one, and the live lanes are a mask.  Fragment starts never move, so
  // each lane's fragment (its lanes, the empty lanes past m joining the last
  // fragment) is fixed for the whole batch.
  const unsigned upto = lane == 31 ? FULL : ((2u << lane) - 1u);  // lanes up to this one
  unsigned alive = m >= 32 ? FULL : ((1u << m) - 1u);
  const unsigned fsm = __ballot_sync(FULL, fst);
  const unsigned before = fsm & upto;
  const int first = before ? 31 - __clz(before) : 0;
  const unsigned after = fsm & ~upto;
  const unsigned fmask = (after ? ((after & (0u - after)) - 1u) : FULL) & ~((1u << first) - 1u);
  for (int step = 0; step <= 32; ++step) {
    const uint32_t k = kr_rank(kr);
    const bool mrg = mergeable(k);  // a retired lane holds KR_WALL
    if (!__any_sync(FULL, mrg)) break;
    if (step == 32) {  // cannot happen: every step merges a pair of some fragment
      if (lane == 0) set_error(st, ST_EINTERNAL);
      break;
    }
    // the fragment's leftmost lowest-rank pair: one reduction over its lanes
    // (every lane takes part, so it comes first)
    const uint32_t v = mrg ? ((k << 5) | (uint32_t)lane) : SEG_VAL;
    const uint32_t fmin = __reduce_min_sync(fmask, v);
    const bool sel = mrg && v == fmin;
    const unsigned selm = __ballot_sync(FULL, sel);
    // neighbours among the live lanes
    const bool live = (alive >> lane) & 1u;
    const unsigned above = alive & ~upto;
    const int nx = above ? __ffs(above) - 1 : 31;            // next live lane
    const unsigned above2 = above & (above - 1u);
    const int nx2 = above2 ? __ffs(above2) - 1 : 31;         // the live lane after it
    const unsigned lower = alive & ((1u << lane) - 1u);
    const bool absorbed = live && lower && ((selm >> (31 - __clz(lower))) & 1u);  // previous live lane merges into it
    const uint32_t res = kr_result(kr);
    const uint32_t sym_nx2 = __shfl_sync(FULL, sym, nx2);
    const uint32_t res_nx = __shfl_sync(FULL, res, nx);
    unsigned long long nkr = kr;
    bool look = false;
    uint32_t la = 0, lb = 0;
    if (sel) {
      sym = res;
      // the merged symbol and the live symbol after the absorbed one
      if (above2 && !((fsm >> nx2) & 1u)) {
        look = true;
        la = res;
        lb = sym_nx2;
      } else {
        nkr = KR_WALL;
      }
    } else if (live && above && ((selm >> nx) & 1u) && !((fsm >> nx) & 1u)) {
      look = true;  // the pair with the merged symbol on the right
      la = sym;
      lb = res_nx;
    }
    if (look) nkr = merge_lookup(V, la, lb);
    if (absorbed) nkr = KR_WALL;
    kr = nkr;
    alive &= ~__ballot_sync(FULL, absorbed);
  }
  // the live symbols, in order, to the first lanes
  const bool live = (alive >> lane) & 1u;
  if (live) {
    const int p = __popc(alive & ((1u << lane) - 1u));
    B.sym[p] = sym;
    B.len[p] = (uint16_t)(fst ? FRAG_START : 0u);
    B.fidx[p] = (uint16_t)fid;
  }
  __syncwarp();
  const int mm = __popc(alive);
  if (lane < mm) {
    sym = B.sym[lane];
    fst = (B.len[lane] & FRAG_START) != 0;
    fid = B.fidx[lane];
  } else {
    sym = 0; fst = false; fid = 0;
  }
  lenb = 0;
  kr = KR_WALL;
  __syncwarp();
  return mm;
}

// One warp encodes a batch of short fragments (at most SB_MAX bytes in all).
__device__ void short_batch(const Call& c, const Workspace& ws, const DevVocab& V, WarpBuf& B, uint8_t* owner,
                            unsigned long long desc) {
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const unsigned long long first = desc >> 5;
  const int nfr = (int)(desc & 31u) + 1;
  const unsigned long long ent = lane < nfr ? ws.sfrag[first + lane] : 0ull;
  const long long start = (long long)(ent >> 8);
  const int len = (int)(ent & 255u);
  int off = len;  // exclusive sum of the lengths over the lanes
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(FULL, off, d);
    if (lane >= d) off += o;
  }
  const int M = __shfl_sync(FULL, off, 31);
  off -= len;
  for (int j = 0; j < len; ++j) owner[off + j] = (uint8_t)lane;
  __syncwarp();
  int fid = lane < M ? owner[lane] : 0;
  __syncwarp();
  const long long fpos = __shfl_sync(FULL, start, fid);
  const int foff = __shfl_sync(FULL, off, fid);
  // batches of short fragments only take the step engine (few merges
  // each, so few steps); a batch with a longer one the sweep engine, which
  // merges all certified-safe pairs at once (monotone vocabularies)
  const unsigned maxlen = __reduce_max_sync(FULL, (unsigned)len);
  const bool stepwise = !V.monotone || maxlen <= STEP_MAX_LEN;
  uint32_t sym = 0, lenb = 0, mlv = 0, mrv = 0;
  bool fst = false;
  if (lane < M) {
    const int j = lane - foff;
    sym = (uint32_t)__ldg(V.byte_id + c.text[fpos + j]);
    lenb = 1;
    fst = j == 0;
    if (!stepwise) {
      mlv = __ldg(V.max_left + sym);
      mrv = __ldg(V.max_right + sym);
    }
  }
  const uint32_t nxt = __shfl_down_sync(FULL, sym, 1);
  const bool nfs = __shfl_down_sync(FULL, fst, 1);
  unsigned long long kr = KR_WALL;
  if (lane + 1 < M && !nfs) kr = merge_lookup(V, sym, nxt);
  const int m = stepwise ? warp_steps(B, V, ws.st, M, sym, lenb, fst, fid, kr)
                         : warp_sweeps(B, V, ws.st, M, sym, lenb, fst, fid, mlv, mrv, kr);
  // ids at the fragment's byte offset, and their number
  const uint32_t fsm = __ballot_sync(FULL, lane < m && fst);
  const long long pos = __shfl_sync(FULL, start, fid);
  if (lane < m) {
    const uint32_t upto = lane == 31 ? 0xffffffffu : ((2u << lane) - 1u);
    const int firstlane = 31 - __clz(fsm & upto);
    ws.tok[pos + (lane - firstlane)] = (int32_t)sym;
    if (fst) {
      const uint32_t after = fsm & ~upto;
      const int nx = after ? __ffs(after) - 1 : m;
      ws.fcnt[pos] = nx - lane;
    }
  }
  // every fragment of a batch starts in the same 512-byte chunk
  if (lane == 0) {
    atomicAdd(&ws.ctot[start / BCHUNK], (uint32_t)m);
    atomicAdd(&ws.gtot[start / BCHUNK / CTOT_GROUP], (uint32_t)m);
  }
  __syncwarp();
}

struct GridParams {         // the grid engine's copy of the kernel parameters
  Call c;
  Workspace ws;
  DevVocab V;
};

// One warp's window of the grid engine's coordinate space for the safe-pair
// walks: GW consecutive coordinates, GW_BEHIND of them before the warp's
// current tile of 32, held as a ring (coordinate p in slot p mod GW).
constexpr int GW = 128;
constexpr int GW_BEHIND = 32;
struct GridWin {
  uint32_t rank[GW];        // rank of the pair (p, next)
  uint32_t sym[GW];
  uint16_t len[GW];
  uint16_t back[GW];
};

struct GridSmem {
  GridParams gp;
  GridWin win[B_THREADS / 32];
};

struct EngineSmem {
  union {
    CtaBatch cb;
    WarpBuf wb[B_THREADS / 32];
    GridSmem g;
  } u;
  uint8_t owner[B_THREADS / 32][SB_MAX];
  int scan[B_THREADS / 32];
  unsigned long long scan64[B_THREADS / 32];
  int sflags;
  uint32_t idx;
  uint32_t nq[3];           // queue sizes: long, 33..B_CAP bytes, short batches
  int gmode;                // the long fragments go to the grid engine
  uint32_t gcnt[B_THREADS / 32];  // grid engine: live symbols of each warp's unit
  unsigned long long end;
};

// End of a long fragment: from its queue entry, or the next fragment start
// after it (or the text end).  All threads of the CTA; the same value in each.
__device__ __forceinline__ long long long_end(const Call& c, const Workspace& ws, const Frag& f,
                                               unsigned long long* send) {
  const int tid = threadIdx.x, T = B_THREADS;
  if (tid == 0) *send = f.len > 0 ? (unsigned long long)(f.start + f.len) : (unsigned long long)c.n;
  __syncthreads();
  if (f.len <= 0) {
    const long long w0 = (f.start + 1) >> 5, wn = (c.n + 31) >> 5;
    for (long long base = w0; base < wn; base += T) {
      const long long wi = base + tid;
      if (wi < wn) {
        uint32_t wv = ws.pstart[wi];
        if (wi == w0) wv &= ~0u << ((f.start + 1) & 31);
        if (wi * 32 + 32 > c.n) wv &= (c.n - wi * 32 >= 32) ? ~0u : ((1u << (c.n - wi * 32)) - 1u);
        if (wv) atomicMin(send, (unsigned long long)(wi * 32 + __ffs(wv) - 1));
      }
      __syncthreads();
      const bool found = *send < (unsigned long long)c.n;
      __syncthreads();
      if (found) break;
    }
  }
  const long long e = (long long)*send;
  __syncthreads();
  return e;
}

// ---------------------------------------------------------------------------
// Grid engine: every fragment longer than B_CAP bytes at once, on the first
// c.grid_ctas CTAs of K3b.  The launch is cooperative, so every CTA of the
// grid is resident and these CTAs can wait for one another at grid barriers.
//
// The fragments lie end to end in one coordinate space, fragment j at
// [o_j, o_j + m_j) in queue order.  A symbol stays at the coordinate of its
// first byte: L[c] is its byte length (0: c lies inside another symbol), the
// next symbol starts at c + L[c] and the previous one at c - B[c] (B[c] = 0:
// c starts its fragment), and K[c] is the key of the pair (c, next), KR_WALL
// at the last symbol of a fragment.  A merge rewrites the two symbols and
// the links of their neighbours only, so nothing is compacted between
// sweeps.  A sweep is the sweep of the global-memory engine (monotone
// vocabularies) in three steps, a grid barrier after each:
//   P1  stale keys are looked up; a mergeable pair whose left neighbour pair
//       is another merge starts a run of equal-rank pairs; live symbols are
//       counted
//   P2  each pair's run start (a max-scan over the whole space: shuffles in a
//       tile, then the last run start of each earlier unit of the group of 32
//       units, then the largest of each earlier group) and its safe flag, the
//       walks reading a per-warp window of the space in shared memory
//   P3  the safe pairs merge
// then each live symbol's rank gives its id's place (grid_ids).  Warp w of
// CTA b owns the coordinates of unit u = 4b + w, [u*R, (u+1)*R) with R a
// multiple of 32, in tiles of 32.  Symbols and links are written by other
// CTAs between barriers, so they are read past L1 (ld.global.cg).  When the
// long fragments hold fewer than GRID_MIN_LONG bytes, the same CTAs take one
// fragment each instead.

constexpr long long GRID_MIN_LONG = 32 * 1024;  // long-fragment bytes from which the grid engine runs
constexpr int GRID_PER_SM = 8;                  // CTAs per SM in the grid engine
constexpr int GRID_UNITS = B_THREADS / 32;      // units (warps) per CTA

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier of the n CTAs of the grid engine; every thread of each CTA calls
// it.  Thread 0 arrives on a counter and, unless it is the last arrival,
// waits for the last one to advance the generation: for at most the call's
// wait limit, after which it marks the call ST_ETIMEOUT and raises the abort
// flag, which ends every other CTA's wait too.  False in every CTA once the
// flag is up.
__device__ bool grid_barrier(const Call& c, DevStatus* st, uint32_t n, int* sflag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const uint32_t gen = ld_acquire(&st->gb_gen);
    __threadfence();
    if (atomicAdd(&st->gb_count, 1u) == n - 1u) {
      atomicExch(&st->gb_count, 0u);
      st_release(&st->gb_gen, gen + 1u);
    } else {
      const unsigned long long t0 = global_ns();
      for (uint32_t it = 0; ld_acquire(&st->gb_gen) == gen; ++it) {
        if (ld_acquire(&st->g_abort) || it >= (1u << 28) || ((it & 31u) == 31u && global_ns() - t0 > c.wait_ns)) {
          atomicExch(&st->g_abort, 1u);
          set_error(st, ST_ETIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
    if (ld_acquire(&st->g_abort)) ok = 0;
    *sflag = ok;
  }
  __syncthreads();
  return *sflag != 0;
}

// The grid engine's symbol arrays (coordinate space of the long fragments).
struct GridSyms {
  uint32_t* S;
  uint16_t* L;
  uint16_t* B;
  unsigned long long* K;
};

// What the safe-pair walks read of the symbol at coordinate p: from the
// warp's window [wlo, wlo + GW) when p lies in it, else from global memory.
struct WinSym {
  uint32_t rank, sym;
  int len, back;
};

__device__ __forceinline__ WinSym win_get(const GridWin& W, long long wlo, long long p, const GridSyms& G) {
  WinSym r;
  const long long d = p - wlo;
  if (d >= 0 && d < GW) {
    const int s = (int)(p & (GW - 1));
    r.rank = W.rank[s];
    r.sym = W.sym[s];
    r.len = W.len[s];
    r.back = W.back[s];
  } else {
    r.rank = kr_rank(__ldcg(G.K + p));
    r.sym = __ldcg(G.S + p);
    r.len = __ldcg(G.L + p);
    r.back = __ldcg(G.B + p);
  }
  return r;
}

// The 32 coordinates [base, base + 32) into the window (one per lane; those
// outside [0, M) are not read).
__device__ __forceinline__ void win_fill(GridWin& W, long long base, long long M, const GridSyms& G) {
  const long long p = base + (threadIdx.x & 31);
  if (p >= 0 && p < M) {
    const int s = (int)(p & (GW - 1));
    W.rank[s] = kr_rank(__ldcg(G.K + p));
    W.sym[s] = __ldcg(G.S + p);
    W.len[s] = __ldcg(G.L + p);
    W.back[s] = __ldcg(G.B + p);
  }
}

// Is the pair at coordinate i (length li of its left symbol, rank k, run
// start u) safe to merge now?  The rule of pair_safe over the linked
// symbols.
__device__ __forceinline__ bool pair_safe_win(const GridWin& W, long long wlo, const GridSyms& G, const DevVocab& V,
                                              long long i, int li, long long u, uint32_t k) {
  const WinSym su = win_get(W, wlo, u, G);
  if (su.back) {
    long long q = u - su.back;
    WinSym sq = win_get(W, wlo, q, G);
    if (sq.rank < k) return false;
    const int lim = V.max_left[su.sym];
    int cum = sq.len;
    while (sq.back) {
      const long long q2 = q - sq.back;
      const WinSym s2 = win_get(W, wlo, q2, G);
      cum += s2.len;
      if (cum > lim) break;
      if (s2.rank < k) return false;
      q = q2;
      sq = s2;
    }
  }
  const long long j1 = i + li;
  const WinSym s1 = win_get(W, wlo, j1, G);
  if (s1.rank != RANK_WALL) {
    if (s1.rank < k) return false;
    const int lim = V.max_right[s1.sym];
    long long q = j1 + s1.len;
    WinSym sq = win_get(W, wlo, q, G);
    int cum = sq.len;
    while (sq.rank != RANK_WALL) {
      const long long q2 = q + sq.len;
      const WinSym s2 = win_get(W, wlo, q2, G);
      cum += s2.len;
      if (cum > lim) break;
      if (sq.rank < k) return false;
      q = q2;
      sq = s2;
    }
  }
  return true;
}

// The grid engine's last steps: each live symbol's rank, then the ids.  A
// function of its own: compiled into the engine, this code costs the rest of
// the kernel registers (measured).
__device__ __noinline__ void grid_ids(uint32_t nlong, EngineSmem& S, long long ulo, long long uhi) {
  const Call& c = S.u.g.gp.c;
  const Workspace& ws = S.u.g.gp.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t P = (uint32_t)c.grid_ctas, nb = P + c.grid_extra, b = blockIdx.x;
  DevStatus* st = ws.st;
  uint32_t* Sy = ws.e_sym[0];
  uint16_t* Ln = ws.e_len[0];
  uint16_t* Bk = ws.e_len[1];
  unsigned long long* K = ws.e_kr[0];
  int32_t* fid = ws.e_rs;
  unsigned long long* off = ws.e_kr[1];
  unsigned long long* fbase = off + nlong + 1;
  long long* urs = reinterpret_cast<long long*>(fbase + nlong);
  unsigned long long* ccnt = reinterpret_cast<unsigned long long*>(urs + (size_t)P * GRID_UNITS);
  // each live symbol's rank (the live counts of the last P1 are final);
  // each fragment's first rank
  unsigned long long pre = 0;
  for (uint32_t y = tid; y < b; y += B_THREADS) pre += __ldcg(ccnt + y);
  unsigned long long cta_pre = 0;
  block_excl_sum64(pre, &cta_pre, S.scan64);
  unsigned long long rank = cta_pre;
  for (int w = 0; w < warp; ++w) rank += S.gcnt[w];
  for (long long t = ulo; t < uhi; t += 32) {
    const long long x = t + lane;
    const bool live = x < uhi && __ldcg(Ln + x) != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, live);
    if (live) {
      const unsigned long long r = rank + __popc(bal & ((1u << lane) - 1u));
      const bool lastsym = kr_rank(__ldcg(K + x)) == RANK_WALL;
      __stcg(K + x, r | (lastsym ? (1ull << 63) : 0ull));
      if (__ldcg(Bk + x) == 0) __stcg(fbase + __ldcg(fid + x), r);
    }
    rank += __popc(bal);
  }
  if (!grid_barrier(c, st, nb, &S.sflags)) return;
  // ids
  for (long long t = ulo; t < uhi; t += 32) {
    const long long x = t + lane;
    if (x < uhi && __ldcg(Ln + x) != 0) {
      const int32_t j = __ldcg(fid + x);
      const long long a = __ldcg(&ws.longq[j].start);
      const unsigned long long kx = __ldcg(K + x);
      const long long k = (long long)((kx & ~(1ull << 63)) - __ldcg(fbase + j));
      ws.tok[a + k] = (int32_t)__ldcg(Sy + x);
      if (kx >> 63) {
        ws.fcnt[a] = (int32_t)(k + 1);
        atomicAdd(&ws.ctot[a / BCHUNK], (uint32_t)(k + 1));
        atomicAdd(&ws.gtot[a / BCHUNK / CTOT_GROUP], (uint32_t)(k + 1));
      }
    }
  }
}

// The long fragments' ids to their byte offsets in ws.tok (and their counts
// to fcnt, ctot and gtot), by the first c.grid_ctas CTAs: all at once when
// they hold GRID_MIN_LONG bytes or more, else one fragment per CTA with the
// global-memory engine.  The arrays are the global-memory engine's: symbols
// e_sym[0], lengths e_len[0], links e_len[1], keys e_kr[0] (after the
// sweeps: each live symbol's rank among all live symbols, bit 63 set at a
// fragment's last), flags e_fl, fragment of each coordinate e_rs; e_kr[1]
// holds the fragment offsets (nlong + 1), the rank of each fragment's first
// symbol (nlong), the last run start of each unit (4 per CTA), the live
// symbols of each CTA and two buffers of the largest run start of each group
// of 32 units.
__device__ __noinline__ void grid_engine(uint32_t nlong, EngineSmem& S) {
  const Call& c = S.u.g.gp.c;
  const Workspace& ws = S.u.g.gp.ws;
  const DevVocab& V = S.u.g.gp.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t P = (uint32_t)c.grid_ctas, nb = P + c.grid_extra, b = blockIdx.x;
  DevStatus* st = ws.st;
  uint32_t* Sy = ws.e_sym[0];
  uint16_t* Ln = ws.e_len[0];
  uint16_t* Bk = ws.e_len[1];
  unsigned long long* K = ws.e_kr[0];
  uint8_t* F = ws.e_fl;
  int32_t* fid = ws.e_rs;
  unsigned long long* off = ws.e_kr[1];
  unsigned long long* fbase = off + nlong + 1;
  long long* urs = reinterpret_cast<long long*>(fbase + nlong);
  unsigned long long* ccnt = reinterpret_cast<unsigned long long*>(urs + (size_t)P * GRID_UNITS);
  const long long ngroups = ((long long)P * GRID_UNITS + 31) / 32;
  long long* ugrp = reinterpret_cast<long long*>(ccnt + P);  // two buffers of ngroups

  // every fragment's length; its id count stays 0 (nothing to emit) unless
  // the engine finishes
  for (uint32_t j = b; j < nlong; j += P) {
    const Frag f = ws.longq[j];
    const long long e = long_end(c, ws, f, &S.end);
    if (tid == 0) {
      ws.longq[j].len = e - f.start;
      ws.fcnt[f.start] = 0;
    }
  }
  if (!grid_barrier(c, st, nb, &S.sflags)) return;
  // their offsets, in queue order: every CTA computes them and stores the
  // same values (no barrier needed before its own reads)
  unsigned long long run = 0;
  for (uint32_t j0 = 0; j0 < nlong; j0 += B_THREADS) {
    const uint32_t j = j0 + tid;
    const unsigned long long m = j < nlong ? (unsigned long long)__ldcg(&ws.longq[j].len) : 0ull;
    unsigned long long tot = 0;
    const unsigned long long ex = block_excl_sum64(m, &tot, S.scan64);
    if (j < nlong) __stcg(off + j, run + ex);
    run += tot;
  }
  if (tid == 0) __stcg(off + nlong, run);
  __syncthreads();
  const long long M = (long long)run;
  if (M < GRID_MIN_LONG) {
    // few long-fragment bytes: one fragment per CTA, fragment j to CTA j mod P
    for (uint32_t j = b; j < nlong; j += P) {
      const long long a = __ldcg(&ws.longq[j].start), m = __ldcg(&ws.longq[j].len);
      const int n = global_engine(c, ws, V, a, (int)m, ws.tok + a, S.scan, S.scan64);
      if (tid == 0) {
        ws.fcnt[a] = n;
        atomicAdd(&ws.ctot[a / BCHUNK], (uint32_t)n);
        atomicAdd(&ws.gtot[a / BCHUNK / CTOT_GROUP], (uint32_t)n);
      }
      __syncthreads();
    }
    return;
  }
  const long long nunits = (long long)P * GRID_UNITS;
  const long long R = ((M + nunits - 1) / nunits + 31) & ~31ll;
  const long long u = (long long)b * GRID_UNITS + warp;
  const long long ulo = min(u * R, M), uhi = min(ulo + R, M);

  // the bytes' symbols
  for (long long t = ulo; t < uhi; t += 32) {
    const long long x = t + lane;
    if (x < uhi) {
      uint32_t lo = 0, hi = nlong;  // off[lo] <= x < off[hi]
      while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        if ((long long)__ldcg(off + mid) <= x) lo = mid;
        else hi = mid;
      }
      const long long o = (long long)__ldcg(off + lo), e = (long long)__ldcg(off + lo + 1);
      const long long a = __ldcg(&ws.longq[lo].start);
      __stcg(Sy + x, (uint32_t)__ldg(V.byte_id + c.text[a + (x - o)]));
      __stcg(Ln + x, (uint16_t)1);
      __stcg(Bk + x, (uint16_t)(x == o ? 0 : 1));
      __stcg(K + x, x + 1 == e ? KR_WALL : KR_NEED);
      __stcg(fid + x, (int32_t)lo);
    }
  }
  if (lane == 0 && (u & 31) == 0) __stcg(ugrp + (u >> 5), -1ll);
  if (!grid_barrier(c, st, nb, &S.sflags)) return;

  for (uint32_t sweep = 0;; ++sweep) {
    // P1: keys, run starts; the live symbols of the unit
    long long last = -1;
    bool any = false;
    uint32_t cnt = 0;
    long long* grp = ugrp + (sweep & 1) * ngroups;
    for (long long t = ulo; t < uhi; t += 32) {
      const long long x = t + lane;
      bool rs = false;
      int l = 0;
      if (x < uhi) {
        l = __ldcg(Ln + x);
        if (l) {
          unsigned long long k = __ldcg(K + x);
          if (kr_rank(k) == RANK_NEED || mergeable(kr_rank(k))) {
            const uint32_t sx = __ldcg(Sy + x), sn = __ldcg(Sy + x + l);
            if (kr_rank(k) == RANK_NEED) {
              k = merge_lookup(V, sx, sn);
              __stcg(K + x, k);
            }
            if (mergeable(kr_rank(k))) {
              any = true;
              const int bx = __ldcg(Bk + x);
              rs = bx == 0 || sn != sx || __ldcg(Sy + x - bx) != sx;
            }
          }
          __stcg(F + x, (uint8_t)(rs ? 2 : 0));
        }
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, rs);
      if (bal) last = t + 31 - __clz(bal);
      cnt += __popc(__ballot_sync(0xffffffffu, l != 0));
    }
    if (lane == 0) {
      __stcg(urs + u, last);
      if (last >= 0) atomicMax(grp + (u >> 5), last);
      // the other buffer, read in the previous sweep, serves the next one
      if ((u & 31) == 0) __stcg(ugrp + ((sweep + 1) & 1) * ngroups + (u >> 5), -1ll);
      S.gcnt[warp] = cnt;
    }
    if (__syncthreads_or(any) && tid == 0) atomicOr(&st->g_any[sweep % 3], 1u);
    if (tid == 0) {
      unsigned long long tot = 0;
      for (int w = 0; w < GRID_UNITS; ++w) tot += S.gcnt[w];
      __stcg(ccnt + b, tot);
    }
    if (b == 0 && tid == 0) atomicExch(&st->g_any[(sweep + 1) % 3], 0u);
    if (!grid_barrier(c, st, nb, &S.sflags)) return;
    if (!ld_acquire(&st->g_any[sweep % 3])) break;
    if (sweep >= (uint32_t)min(M, 1ll << 30)) {
      if (tid == 0) set_error(st, ST_EINTERNAL);
      return;
    }
    // P2: run starts, safe flags.  The run start carried into the unit:
    // the last one of the nearest earlier unit of its group of 32 units
    // that has one, else the largest of the nearest earlier group that has
    // one
    long long carry = -1;
    if (ulo < uhi) {
      const long long g = u >> 5, v = u - 1 - lane;
      long long r = v >= (g << 5) ? __ldcg(urs + v) : -1ll;
      uint32_t hit = __ballot_sync(0xffffffffu, r >= 0);
      for (long long g0 = g - 1; !hit && g0 >= 0; g0 -= 32) {
        const long long gg = g0 - lane;
        r = gg >= 0 ? __ldcg(grp + gg) : -1ll;
        hit = __ballot_sync(0xffffffffu, r >= 0);
      }
      if (hit) carry = __shfl_sync(0xffffffffu, r, __ffs(hit) - 1);
    }
    // the warp's window: [wlo, wlo + GW) around its current tile
    GridWin& W = S.u.g.win[warp];
    const GridSyms G{Sy, Ln, Bk, K};
    long long wlo = ulo - GW_BEHIND;
    if (ulo < uhi) {
#pragma unroll
      for (int q = 0; q < GW / 32; ++q) win_fill(W, wlo + 32 * q, M, G);
      __syncwarp();
    }
    for (long long t = ulo; t < uhi; t += 32) {
      const long long x = t + lane;
      int l = 0, f = 0;
      uint32_t kr = RANK_WALL;
      if (x < uhi) {
        const int s = (int)(x & (GW - 1));
        l = W.len[s];
        if (l) {
          f = __ldcg(F + x);
          kr = W.rank[s];
        }
      }
      long long rsx = (f & 2) ? x : -1ll;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, rsx, o);
        if (lane >= o) rsx = max(rsx, y);
      }
      rsx = max(rsx, carry);
      carry = __shfl_sync(0xffffffffu, rsx, 31);
      if (l) {
        bool safe = false;
        if (mergeable(kr)) {
          // pairs of a run alternate from its start; the run's symbols all
          // have this symbol's length
          const unsigned long long d = (unsigned long long)(x - rsx);
          const unsigned long long q = d < 0x80000000ull ? (unsigned long long)((uint32_t)d / (uint32_t)l)
                                                         : d / (unsigned long long)l;
          safe = !(q & 1ull) && pair_safe_win(W, wlo, G, V, x, l, rsx, kr);
        }
        __stcg(F + x, (uint8_t)(safe ? 1 : 0));
      }
      // slide the window by one tile
      __syncwarp();
      win_fill(W, wlo + GW, M, G);
      wlo += 32;
      __syncwarp();
    }
    if (!grid_barrier(c, st, nb, &S.sflags)) return;
    // P3: merges
    for (long long t = ulo; t < uhi; t += 32) {
      const long long x = t + lane;
      if (x < uhi) {
        const int l = __ldcg(Ln + x);
        if (l && (__ldcg(F + x) & 1)) {
          const long long j = x + l;
          const int lj = __ldcg(Ln + j);
          const bool wall = kr_rank(__ldcg(K + j)) == RANK_WALL;
          const int nl = l + lj;
          __stcg(Sy + x, kr_result(__ldcg(K + x)));
          __stcg(Ln + x, (uint16_t)nl);
          __stcg(Ln + j, (uint16_t)0);
          __stcg(K + x, wall ? KR_WALL : KR_NEED);
          if (!wall) __stcg(Bk + j + lj, (uint16_t)nl);
          const int bx = __ldcg(Bk + x);
          if (bx) __stcg(K + x - bx, KR_NEED);
        }
      }
    }
    if (!grid_barrier(c, st, nb, &S.sflags)) return;
  }

  grid_ids(nlong, S, ulo, uhi);
}

// K3b: a persistent grid.  Longest work first: fragments of more than B_CAP
// bytes (the grid engine's CTAs, or every CTA taking one at a time for the
// global-memory engine), then those of 33..B_CAP bytes (shared-memory
// engine, one fragment per CTA), then batches of short fragments (warp step
// or sweep engine, one batch per warp, counted from the other end of the
// grid so that the CTAs with a 33..B_CAP-byte fragment get fewer).  Static
// assignment keeps thousands of warps off one contended counter.
// GRID: the grid engine is compiled in (the launch is then cooperative);
// without it the kernel carries no call, whose calling convention costs the
// other paths registers.
template <bool GRID>
__global__ void __launch_bounds__(B_THREADS, 16) k_bpe_engine(Call c, Workspace ws, DevVocab V) {
  __shared__ EngineSmem S;
  const int tid = threadIdx.x, warp = tid >> 5, T = B_THREADS;
  // launched as a programmatic dependent of the boundary kernel: wait until
  // it has completed and its writes are visible; let the emit kernel's CTAs
  // be scheduled as this grid's retire
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  DevStatus* st = ws.st;
  if (tid == 0) {  // the queue sizes, loaded together (K2 wrote them)
    S.nq[0] = st->long_count;
    S.nq[1] = st->wide_count;
    S.nq[2] = st->sbatch_count;
  }
  __syncthreads();
  const uint32_t nlong = S.nq[0];
  // Where the grid engine can run, CTAs [0, c0) take the long fragments
  // (all at once when they hold many bytes, else one each) and nothing else;
  // CTAs [c0, grid) take the other queues.  Else every CTA takes long
  // fragments one at a time, then the other queues.
  const uint32_t c0 = GRID && nlong && V.monotone && c.grid_ctas > 0 ? (uint32_t)c.grid_ctas : 0u;
  if (GRID && c0) {
#pragma nv_diag_suppress 186  // without GRID, c0 is the constant 0
    if (blockIdx.x < c0) {
#pragma nv_diag_default 186
      if (tid == 0) {
        S.u.g.gp.c = c;
        S.u.g.gp.ws = ws;
        S.u.g.gp.V = V;
      }
      __syncthreads();
      grid_engine(nlong, S);
      return;
    }
  } else {
    while (nlong) {
      // one thread decides for the CTA (the loop has barriers); the plain
      // read first keeps CTAs without work off the contended counter
      if (tid == 0)
        S.idx = *(volatile const uint32_t*)&st->long_taken < nlong ? atomicAdd(&st->long_taken, 1u) : nlong;
      __syncthreads();
      const uint32_t idx = S.idx;
      __syncthreads();
      if (idx >= nlong) break;
      const Frag f = ws.longq[idx];
      const long long a = f.start;
      const long long e = long_end(c, ws, f, &S.end);
      const int m = global_engine(c, ws, V, a, (int)(e - a), ws.tok + a, S.scan, S.scan64);
      if (tid == 0) {
        ws.fcnt[a] = m;
        atomicAdd(&ws.ctot[a / BCHUNK], (uint32_t)m);
        atomicAdd(&ws.gtot[a / BCHUNK / CTOT_GROUP], (uint32_t)m);
      }
      __syncthreads();
    }
  }
  const uint32_t G = gridDim.x - c0, bb = blockIdx.x - c0;
  const uint32_t nwide = S.nq[1];
  for (uint32_t i = bb; i < nwide; i += G) {
    const Frag f = ws.wq[i];
    cta_fragment(c, ws, V, f.start, (int)f.len, S.u.cb, S.scan, S.scan64, &S.sflags);
  }
  __syncthreads();
  const uint32_t nbat = S.nq[2];
  const uint32_t nwarps = G * (T / 32);
  const uint32_t gw = (G - 1 - bb) * (T / 32) + warp;
  // one batch per warp first (no counter); with more batches than warps the
  // rest go to whichever warp is free, each claim issued before the batch
  // in hand runs, so that its latency hides behind that batch
  const bool claim = nbat > nwarps;
  uint32_t b = gw;
  while (b < nbat) {
    uint32_t nx = 0;
    if (claim && (threadIdx.x & 31) == 0) nx = nwarps + atomicAdd(&st->sbatch_taken, 1u);
    short_batch(c, ws, V, S.u.wb[warp], S.owner[warp], ws.sbatch[b]);
    if (!claim) break;
    b = __shfl_sync(0xffffffffu, nx, 0);
  }
}

void launch_bpe_engine(const Call& call, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  // a persistent grid of as many CTAs as fit at once (16 of 32 registers per
  // SM), launched as a programmatic dependent of the boundary kernel (its
  // CTAs are scheduled while that grid's last CTAs finish) and, where the
  // grid engine can run (a monotone vocabulary, a text of GRID_MIN_LONG bytes
  // or more), cooperatively: all CTAs resident together, as the grid
  // engine's CTAs wait for one another
  constexpr int kMaxDev = 64;
  static int per_sm[kMaxDev] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int& ps = per_sm[dev >= 0 && dev < kMaxDev ? dev : 0];
  if (!ps) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_bpe_engine<true>, B_THREADS, 0) != cudaSuccess) {
      cudaGetLastError();
      occ = 1;
    }
    ps = occ < 1 ? 1 : (occ > 16 ? 16 : occ);
  }
  const unsigned long long grid = (unsigned long long)n_sms * ps;
  Call c = call;
  // the grid engine keeps in e_kr[1] two words per long fragment and one
  // more, then per CTA one word per unit, one for the CTA and two buffers of
  // one word per 32 units (at most 2 + 1 per CTA with GRID_UNITS <= 16)
  static_assert(GRID_UNITS <= 16, "two group words per CTA at most");
  const unsigned long long lq = w.cap_bytes / (B_CAP + 1) + w.cap_bytes / BCHUNK + 256;
  const unsigned long long words = w.cap_bytes + 256;
  const unsigned long long room = words > 2 * lq + 3 ? (words - 2 * lq - 3) / (GRID_UNITS + 2) : 0;
  unsigned long long gc = (unsigned long long)n_sms * (ps < GRID_PER_SM ? ps : GRID_PER_SM);
  if (gc > room) gc = room;
  if (gc + 1 > grid) gc = grid - 1;
  if (c.n < GRID_MIN_LONG || !v.monotone) gc = 0;  // the grid engine cannot run
  c.grid_ctas = (int)gc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(B_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  // cooperative only where the grid engine may wait at its barriers
  cfg.numAttrs = gc ? 2 : 1;
  if (gc) cudaLaunchKernelEx(&cfg, k_bpe_engine<true>, c, w, v);
  else cudaLaunchKernelEx(&cfg, k_bpe_engine<false>, c, w, v);
}

}  // namespace tokgb
