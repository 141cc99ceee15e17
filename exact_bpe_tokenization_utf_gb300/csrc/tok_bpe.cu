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
    if (sweep == m0 && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);
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
  for (int i = tid; i < M; i += T) C.kr[i] = (i + 1 >= M) ? KR_WALL : merge_lookup(V, C.sym[i], C.sym[i + 1]);
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
        if (jn >= m) nkr[j] = KR_WALL;
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
    if (sweep == M && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);  // cannot happen: every sweep merges
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
      if (lane == 0) atomicExch(&st->code, ST_EINTERNAL);
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
      if (lane == 0) atomicExch(&st->code, ST_EINTERNAL);
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

struct EngineSmem {
  union {
    CtaBatch cb;
    WarpBuf wb[B_THREADS / 32];
  } u;
  uint8_t owner[B_THREADS / 32][SB_MAX];
  int scan[B_THREADS / 32];
  unsigned long long scan64[B_THREADS / 32];
  int sflags;
  uint32_t idx;
  uint32_t nq[3];           // queue sizes: long, 33..B_CAP bytes, short batches
  unsigned long long end;
};

// K3b: a persistent grid.  Longest work first: fragments of more than B_CAP
// bytes (global-memory engine, taken one at a time), then those of 33..B_CAP
// bytes (shared-memory engine, fragment i to CTA i mod grid), then batches of
// short fragments (warp step or sweep engine, batch b to warp b mod warps,
// counted from the last CTA so that the CTAs with a 33..B_CAP-byte fragment
// get fewer).
// Static assignment keeps thousands of warps off one contended counter.
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
  while (nlong) {
    // one thread decides for the CTA (the loop has barriers); the plain read
    // first keeps CTAs without work off the contended counter
    if (tid == 0)
      S.idx = *(volatile const uint32_t*)&st->long_taken < nlong ? atomicAdd(&st->long_taken, 1u) : nlong;
    __syncthreads();
    const uint32_t idx = S.idx;
    __syncthreads();
    if (idx >= nlong) break;
    const Frag f = ws.longq[idx];
    // end: known from the queue entry, or the next fragment start after
    // f.start (or the text end)
    if (tid == 0) S.end = f.len > 0 ? (unsigned long long)(f.start + f.len) : (unsigned long long)c.n;
    __syncthreads();
    if (f.len <= 0) {
      const long long w0 = (f.start + 1) >> 5, wn = (c.n + 31) >> 5;
      for (long long base = w0; base < wn; base += T) {
        const long long wi = base + tid;
        if (wi < wn) {
          uint32_t wv = ws.pstart[wi];
          if (wi == w0) wv &= ~0u << ((f.start + 1) & 31);
          if (wi * 32 + 32 > c.n) wv &= (c.n - wi * 32 >= 32) ? ~0u : ((1u << (c.n - wi * 32)) - 1u);
          if (wv) atomicMin(&S.end, (unsigned long long)(wi * 32 + __ffs(wv) - 1));
        }
        __syncthreads();
        const bool found = S.end < (unsigned long long)c.n;
        __syncthreads();
        if (found) break;
      }
    }
    const long long a = f.start;
    const int m = global_engine(c, ws, V, a, (int)((long long)S.end - a), ws.tok + a, S.scan, S.scan64);
    if (tid == 0) {
      ws.fcnt[a] = m;
      atomicAdd(&ws.ctot[a / BCHUNK], (uint32_t)m);
      atomicAdd(&ws.gtot[a / BCHUNK / CTOT_GROUP], (uint32_t)m);
    }
    __syncthreads();
  }
  const uint32_t nwide = S.nq[1];
  for (uint32_t i = blockIdx.x; i < nwide; i += gridDim.x) {
    const Frag f = ws.wq[i];
    cta_fragment(c, ws, V, f.start, (int)f.len, S.u.cb, S.scan, S.scan64, &S.sflags);
  }
  __syncthreads();
  const uint32_t nbat = S.nq[2];
  const uint32_t nwarps = gridDim.x * (T / 32);
  const uint32_t gw = (gridDim.x - 1 - blockIdx.x) * (T / 32) + warp;
  for (uint32_t b = gw; b < nbat; b += nwarps) short_batch(c, ws, V, S.u.wb[warp], S.owner[warp], ws.sbatch[b]);
}


void launch_bpe_engine(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  // 16 CTAs of 32 registers per SM; a programmatic dependent of the boundary
  // kernel (its CTAs are scheduled while that grid's last CTAs finish)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_sms * 16));
  cfg.blockDim = dim3(B_THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, k_bpe_engine, c, w, v);
}

}  // namespace tokgb
