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
// K3: the fragments that start in one 512-byte chunk
//
// Most fragments need no merge loop: a single byte is its byte token, and a
// fragment whose bytes equal a token t with BPE(bytes(t)) == [t] (checked for
// every token at load time) encodes to [t].  Each thread settles a few
// fragments with one hash probe each, all its probes issued before it waits.
// The rest are encoded by one of three engines, all running the same sweep
// (every certified-safe pair merges):
//   - fragments of at most 32 bytes, packed in order into batches of at most
//     32 symbols, one batch per warp at a time: one symbol per lane,
//     neighbours through shuffles, walls between fragments, no block barrier;
//   - fragments of 33..B_CAP bytes: the whole CTA, in shared memory;
//   - the one fragment longer than B_CAP a chunk can hold besides its last
//     (two such would not both start within 512 bytes): the whole CTA, with
//     the global-memory engine.
// Engine results go to a per-byte scratch array at their fragment's offset
// and are compacted into the chunk's ids at the end.

constexpr int K3_WARPS = K3_THREADS / 32;
constexpr int S_MAX = BCHUNK / 2 + 1;        // unresolved fragments of >= 2 bytes starting in a chunk
constexpr int U_MAX = BCHUNK / 33 + 2;       // fragments of more than 32 bytes starting in a chunk

struct WarpBuf {            // one warp's compaction buffer
  uint32_t sym[32];
  unsigned long long kr[32];
  uint16_t len[32];         // byte length | FRAG_START
  uint16_t fidx[32];
  uint16_t ml[32];
  uint16_t mr[32];
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

struct ChunkEngine {
  union {
    WarpBuf wb[K3_WARPS];
    CtaBatch cb;
  } u;
  // the CTA's bytes and fragment starts
  uint8_t text[B_RANGE];
  uint32_t bits[B_RANGE / 32];
  // fragments that start in the chunk (at most BCHUNK)
  uint16_t fstart[BCHUNK + 1];  // relative to `first`; then the span
  int32_t ftok[BCHUNK];         // settled token, or -1
  uint16_t fcnt[BCHUNK];        // ids of each fragment
  uint16_t fout[BCHUNK];        // first id of each fragment
  uint16_t feng[BCHUNK];        // first CTA-engine symbol of a fragment in its batch
  uint16_t slist[S_MAX];        // unresolved fragments of <= 32 bytes, in order
  uint16_t soff[S_MAX + 1];     // their byte offsets among themselves, then the total
  uint16_t sbat[S_MAX + 1];     // first slist entry of each warp batch, then ns
  uint16_t ulist[U_MAX];        // unresolved fragments of 33..B_CAP bytes, in order
  uint16_t ueoff[U_MAX + 1];    // their byte offsets among themselves, then the total
  int scan[K3_WARPS];
  unsigned long long scan64[K3_WARPS];
  long long first, end, longfrag, item0;
  int nf, ns, nu, nb, sflags, batch_end, big;
};

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
      // a lower rank further away: walk the length-bounded windows
      if (__any_sync(FULL, need)) {
        bool ok = need;
        // left: a token grown from pair q <= u-2 ends at symbol u-1
        int cum = (int)__shfl_sync(FULL, lenb, max(u - 1, 0));
        bool done = !(need && has_l && u >= 2);
        for (int step = 2; step < 32; ++step) {
          const int q = u - step;
          const uint32_t kq = __shfl_sync(FULL, k, max(q, 0));
          const int lq = (int)__shfl_sync(FULL, lenb, max(q, 0));
          if (!done) {
            if (q < 0 || kq == RANK_WALL) done = true;
            else {
              cum += lq;
              if (cum > (int)ml_u) done = true;
              else if (kq < k) { ok = false; done = true; }
            }
          }
          if (!__any_sync(FULL, !done)) break;
        }
        // right: a token grown from pair q >= i+2 starts at symbol i+2
        cum = (int)__shfl_sync(FULL, lenb, min(lane + 2, 31));
        done = !(need && ok && has_r);
        for (int step = 2; step < 32; ++step) {
          const int q = lane + step;
          const uint32_t kq = __shfl_sync(FULL, k, min(q, 31));
          const int lq = (int)__shfl_sync(FULL, lenb, min(q + 1, 31));
          if (!done) {
            if (q > 31 || kq == RANK_WALL) done = true;
            else {
              cum += lq;
              if (cum > (int)mr_i1) done = true;
              else if (kq < k) { ok = false; done = true; }
            }
          }
          if (!__any_sync(FULL, !done)) break;
        }
        if (need) safe = ok;
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

// One warp encodes the short fragments slist[s0..s1) (at most 32 bytes in all).
__device__ void warp_batch(ChunkEngine& E, WarpBuf& B, const Call& c, const DevVocab& V, DevStatus* st,
                           uint32_t* eres, long long fs, int s0, int s1) {
  const int lane = threadIdx.x & 31;
  const unsigned FULL = 0xffffffffu;
  const int base = E.soff[s0];
  const int M = E.soff[s1] - base;
  uint32_t sym = 0, lenb = 0, mlv = 0, mrv = 0;
  bool fst = false;
  int fid = 0;
  if (lane < M) {
    int a = s0, b = s1 - 1;  // entry with soff[a] <= base + lane < soff[a+1]
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (E.soff[mid] <= base + lane) a = mid; else b = mid - 1;
    }
    fid = E.slist[a];
    const int j = base + lane - E.soff[a];
    const int32_t id = __ldg(V.byte_id + E.text[E.fstart[fid] + j]);
    sym = (uint32_t)id;
    lenb = 1;
    fst = j == 0;
    mlv = __ldg(V.max_left + id);
    mrv = __ldg(V.max_right + id);
  }
  const uint32_t nxt = __shfl_down_sync(FULL, sym, 1);
  const bool nfs = __shfl_down_sync(FULL, fst, 1);
  unsigned long long kr = KR_WALL;
  if (lane + 1 < M && !nfs) kr = merge_lookup(V, sym, nxt);
  const int m = warp_sweeps(B, V, st, M, sym, lenb, fst, fid, mlv, mrv, kr);
  // ids to the scratch at the fragment's byte offset, and their number
  const uint32_t fsm = __ballot_sync(FULL, lane < m && fst);
  if (lane < m) {
    const uint32_t upto = lane == 31 ? 0xffffffffu : ((2u << lane) - 1u);
    const int first = 31 - __clz(fsm & upto);
    eres[fs + E.fstart[fid] + (lane - first)] = sym;
    if (fst) {
      const uint32_t after = fsm & ~upto;
      const int nx = after ? __ffs(after) - 1 : m;
      E.fcnt[fid] = (uint16_t)(nx - lane);
    }
  }
}

// 228 KB of shared memory per SM less 1 KB reserved per CTA: at least 8 CTAs
static_assert(8 * (sizeof(ChunkEngine) + 1024) <= 228 * 1024, "K3 shared memory exceeds 8 CTAs per SM");

__global__ void __launch_bounds__(K3_THREADS) k_bpe_chunk(Call c, Workspace ws, DevVocab V) {
  extern __shared__ __align__(16) uint8_t dsm[];
  ChunkEngine& E = *reinterpret_cast<ChunkEngine*>(dsm);
  const int tid = threadIdx.x, T = K3_THREADS, lane = tid & 31, warp = tid >> 5;
  const long long chunk = blockIdx.x;
  const long long r0 = chunk * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  const long long lim = min(r0 + B_RANGE, c.n);
  if (tid < B_RANGE / 32) {
    const long long p = r0 + 32ll * tid;
    uint32_t v = 0;
    if (p < lim) {
      v = ws.pstart[(r0 >> 5) + tid];
      if (lim - p < 32) v &= (1u << (lim - p)) - 1u;
    }
    E.bits[tid] = v;
  }
  if (tid == 0) {
    E.sflags = 0;
    E.big = -1;
  }
  __syncthreads();
  if (tid < 32) {
    // first and last fragment start in [r0, r1) (words 0..15), first start in [r1, lim) (16..23)
    const uint32_t w = lane < B_RANGE / 32 ? E.bits[lane] : 0u;
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
  // settle single bytes and whole tokens: at most 4 fragments per thread,
  // every first probe issued before any is used
  const int FB = (nf + T - 1) / T;
  const int flo = min(tid * FB, nf), fhi = min(flo + FB, nf);
  {
    unsigned long long h[4];
    uint32_t slot[4];
    uint4 e[4];
    int fa[4], fL[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = flo + q;
      fa[q] = 0; fL[q] = 0; h[q] = 0; slot[q] = 0;
      e[q] = make_uint4(0u, 0u, 0u, 0u);
      if (f < fhi) {
        fa[q] = E.fstart[f];
        fL[q] = E.fstart[f + 1] - fa[q];
        if (fL[q] > 1 && whole_eligible(V, fL[q])) {
          h[q] = bytes_hash(E.text + fa[q], fL[q]);
          slot[q] = whole_first_slot(V, h[q]);
          e[q] = __ldg(reinterpret_cast<const uint4*>(V.whole + slot[q]));
        }
      }
    }
    int scount = 0, ucount = 0, sbytes = 0, ubytes = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int f = flo + q;
      if (f < fhi) {
        const int L = fL[q];
        int t = -1;
        if (L == 1) t = __ldg(V.byte_id + E.text[fa[q]]);
        else if (whole_eligible(V, L)) t = whole_lookup_at(V, E.text + fa[q], L, h[q], slot[q], e[q]);
        E.ftok[f] = t;
        E.fcnt[f] = t >= 0 ? 1 : 0;
        if (t < 0) {
          if (L <= 32) { ++scount; sbytes += L; }
          else if (L <= B_CAP) { ++ucount; ubytes += L; }
          else E.big = f;  // at most one per chunk
        }
      }
    }
    int ns = 0, nu = 0, sb_all = 0, ub_all = 0;
    int si = block_excl_sum(scount, &ns, E.scan);
    int so = block_excl_sum(sbytes, &sb_all, E.scan);
    int ui = block_excl_sum(ucount, &nu, E.scan);
    int uo = block_excl_sum(ubytes, &ub_all, E.scan);
    for (int f = flo; f < fhi; ++f) {
      if (E.ftok[f] >= 0) continue;
      const int L = E.fstart[f + 1] - E.fstart[f];
      if (L <= 32) {
        E.slist[si] = (uint16_t)f;
        E.soff[si] = (uint16_t)so;
        ++si;
        so += L;
      } else if (L <= B_CAP) {
        E.ulist[ui] = (uint16_t)f;
        E.ueoff[ui] = (uint16_t)uo;
        ++ui;
        uo += L;
      }
    }
    if (tid == 0) {
      E.soff[ns] = (uint16_t)sb_all;
      E.ueoff[nu] = (uint16_t)ub_all;
      E.ns = ns;
      E.nu = nu;
    }
  }
  __syncthreads();
  // short fragments: greedy batches of at most 32 bytes, in order
  if (tid == 0) {
    const int ns = E.ns;
    int nb = 0, k = 0;
    while (k < ns) {
      E.sbat[nb++] = (uint16_t)k;
      const int b0 = E.soff[k];
      ++k;
      while (k < ns && E.soff[k + 1] - b0 <= 32) ++k;
    }
    E.sbat[nb] = (uint16_t)ns;
    E.nb = nb;
  }
  __syncthreads();
  uint32_t* const eres = ws.e_sym[0];  // engine results, at their fragment's byte offset
  {
    const int nb = E.nb;
    for (int b = warp; b < nb; b += K3_WARPS) warp_batch(E, E.u.wb[warp], c, V, ws.st, eres, fs, E.sbat[b], E.sbat[b + 1]);
  }
  __syncthreads();
  // fragments of 33..B_CAP bytes: CTA engine batches
  const int nu = E.nu;
  CtaBatch& C = E.u.cb;
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
      const int32_t id = __ldg(V.byte_id + E.text[E.fstart[f] + j]);
      C.sym[i] = (uint32_t)id;
      C.len[i] = (uint16_t)(1u | (j == 0 ? FRAG_START : 0u));
      C.fidx[i] = (uint16_t)f;
      C.ml[i] = __ldg(V.max_left + id);
      C.mr[i] = __ldg(V.max_right + id);
    }
    __syncthreads();
    for (int i = tid; i < M; i += T)
      C.kr[i] = (i + 1 >= M || (C.len[i + 1] & FRAG_START)) ? KR_WALL : merge_lookup(V, C.sym[i], C.sym[i + 1]);
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
      if (lane == 0 && fl2) atomicOr(&E.sflags, fl2);
      __syncthreads();
      const int flags = E.sflags;
      if (!(flags & 1)) break;
      if (flags & 2) {
        int lastrun = -1;
        for (int i = lo; i < hi; ++i)
          if (i == 0 || kr_rank(C.kr[i - 1]) != kr_rank(C.kr[i])) lastrun = i;
        int run = block_excl_max(lastrun, E.scan);
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
        best = block_min_u64(best, E.scan64);
        for (int i = lo; i < hi; ++i) C.fl[i] = ((uint32_t)best == (uint32_t)i) ? 1 : 0;
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
          nfi[j] = C.fidx[i];
          const int jn = mg ? i + 2 : i + 1;  // the next symbol that survives
          if (jn >= m || (C.len[jn] & FRAG_START)) nkr[j] = KR_WALL;
          else if (!mg && !C.fl[jn]) nkr[j] = C.kr[i];  // unchanged pair keeps its key
          else nkr[j] = merge_lookup(V, nsym[j], C.fl[jn] ? kr_result(C.kr[jn]) : C.sym[jn]);
        }
      }
      int newm = 0;
      const int bpos = block_excl_sum(__popc(keep), &newm, E.scan);
#pragma unroll
      for (int j = 0; j < B_EPT; ++j) {
        if ((keep >> j) & 1u) {
          const int p = bpos + __popc(keep & ((1u << j) - 1u));
          C.sym[p] = nsym[j];
          C.len[p] = nlen[j];
          C.kr[p] = nkr[j];
          C.fidx[p] = nfi[j];
          C.ml[p] = nml[j];
          C.mr[p] = nmr[j];
        }
      }
      if (tid == 0) E.sflags = 0;
      m = newm;
      __syncthreads();
      if (sweep == M && tid == 0) atomicExch(&ws.st->code, ST_EINTERNAL);  // cannot happen: every sweep merges
    }
    // this batch's results: ids per fragment, symbols to the per-byte scratch
    for (int i = tid; i < m; i += T)
      if (C.len[i] & FRAG_START) E.feng[C.fidx[i]] = (uint16_t)i;
    __syncthreads();
    for (int k = ub + tid; k < ue; k += T) {
      const int f = E.ulist[k];
      const int nx = (k + 1 < ue) ? E.feng[E.ulist[k + 1]] : m;
      E.fcnt[f] = (uint16_t)(nx - E.feng[f]);
    }
    for (int i = tid; i < m; i += T) {
      const int f = C.fidx[i];
      eres[fs + E.fstart[f] + (i - E.feng[f])] = C.sym[i];
    }
    if (tid == 0) E.sflags = 0;
    __syncthreads();
    ub = ue;
  }
  // an unresolved fragment longer than a batch holds
  const int big = E.big;
  if (big >= 0) {
    const long long a = fs + E.fstart[big];
    const int L = E.fstart[big + 1] - E.fstart[big];
    const int m = global_engine(c, ws, V, a, L, reinterpret_cast<int32_t*>(eres) + a, E.scan, E.scan64);
    if (tid == 0) E.fcnt[big] = (uint16_t)m;
    __syncthreads();
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
      const long long e0 = fs + E.fstart[f];
      const int cnt = E.fcnt[f];
      for (int j = 0; j < cnt; ++j) ws.tok[fs + o + j] = (int32_t)eres[e0 + j];
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
// K4: the queued long last fragments of chunks, one CTA each, with the
// global-memory engine; ids at the fragment's byte offset

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
    const int m = global_engine(c, ws, V, a, (int)((long long)s_end - a), ws.tok + a, sh, sh64);
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
  k_bpe_chunk<<<(unsigned)n_bchunks(c.n), K3_THREADS, sizeof(ChunkEngine), s>>>(c, w, v);
}

void launch_bpe_long(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_long<<<n_sms, LONG_THREADS, 0, s>>>(c, w, v);
}

}  // namespace tokgb
