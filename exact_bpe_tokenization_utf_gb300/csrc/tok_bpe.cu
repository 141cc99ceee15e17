// Per-fragment BPE, E ("TokTier: exact stateful tokenization for agentic LLM
// serving", Section 4.2): every fragment is encoded on its own by merging the
// lowest-rank adjacent pair (leftmost on ties) until no adjacent pair is a
// merge.  The pages tier fragments by length (one thread, one warp, one block
// per fragment); here a fragment is settled by one probe when it is a single
// byte or a whole self-encoding token; otherwise it gets one lane per symbol
// in a segment of 8, 16 or 32 lanes (<= 32 bytes), a share of a warp batch
// (<= 128 bytes), or a CTA (longer).
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
// K3: settle the fragments that start in one 512-byte chunk
//
// Most fragments need no merge loop: a single byte is its byte token, and a
// fragment whose bytes equal a token t with BPE(bytes(t)) == [t] (checked for
// every token at load time) encodes to [t].  One thread per fragment settles
// those with a hash probe; the others are queued by length for K3b (segment
// engine up to 32 bytes, warp engine up to WCAP bytes) or K4.

__global__ void __launch_bounds__(B_THREADS) k_settle(Call c, Workspace ws, DevVocab V) {
  __shared__ __align__(16) uint8_t text[S_RANGE];
  __shared__ uint32_t bits[S_RANGE / 32];
  __shared__ uint16_t fstart[BCHUNK + 1];
  __shared__ int scan[B_THREADS / 32];
  __shared__ long long s_last_end;
  __shared__ uint32_t s_qbase[5];
  __shared__ unsigned long long scan64[B_THREADS / 32];
  const int tid = threadIdx.x, T = B_THREADS;
  const long long r0 = (long long)blockIdx.x * BCHUNK;
  const long long r1 = min(r0 + BCHUNK, c.n);
  const long long lim = min(r0 + S_RANGE, c.n);
  const int nb = (int)(lim - r0);
  if (((reinterpret_cast<uintptr_t>(c.text) & 15u) == 0) && nb == S_RANGE) {
    for (int k = tid; k < S_RANGE / 16; k += T)
      reinterpret_cast<uint4*>(text)[k] = reinterpret_cast<const uint4*>(c.text + r0)[k];
  } else {
    for (int k = tid; k < nb; k += T) text[k] = c.text[r0 + k];
  }
  if (tid < S_RANGE / 32) {
    const long long p = r0 + 32ll * tid;
    uint32_t v = 0;
    if (p < lim) {
      v = ws.pstart[(r0 >> 5) + tid];
      if (lim - p < 32) v &= (1u << (lim - p)) - 1u;
    }
    bits[tid] = v;
  }
  __syncthreads();
  if (tid == 0) {  // end of the last fragment: the first start at or after r1
    long long e = -1;
    if (r1 >= c.n) {
      e = c.n;
    } else {
      for (int w = BCHUNK / 32; w < S_RANGE / 32 && e < 0; ++w)
        if (bits[w]) e = r0 + 32ll * w + (__ffs(bits[w]) - 1);
      if (e < 0 && lim >= c.n) e = c.n;
    }
    s_last_end = e;
  }
  // fragment starts in [r0, r1): thread t looks at 4 bit positions
  const int q0 = tid * 4;
  const uint32_t mine = (bits[q0 >> 5] >> (q0 & 31)) & 0xFu;
  int nf = 0;
  int idx = block_excl_sum(__popc(mine), &nf, scan);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if ((mine >> q) & 1u) fstart[idx++] = (uint16_t)(q0 + q);
  __syncthreads();
  // contiguous blocks of at most 4 fragments per thread (nf <= BCHUNK = 4 * T)
  const int FB = (nf + T - 1) / T;
  const int flo = min(tid * FB, nf), fhi = min(flo + FB, nf);
  int qcls[4];                                // queue of each of this thread's fragments, or -1
  long long flen[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int f = flo + j;
    flen[j] = 0;
    qcls[j] = -1;
    if (f >= fhi) continue;
    const int a = fstart[f];
    const long long e = (f + 1 < nf) ? r0 + fstart[f + 1] : s_last_end;
    const long long L = e < 0 ? -1 : e - (r0 + a);
    flen[j] = L;
    int t = -1;
    if (L == 1) t = V.byte_id[text[a]];
    else if (L > 1 && a + L <= S_RANGE) t = whole_lookup(V, text + a, (int)L);
    if (t >= 0) {
      ws.tok[r0 + a] = t;
      ws.fcnt[r0 + a] = 1;
    } else {
      qcls[j] = (L > 1 && L <= 8) ? 0 : (L > 1 && L <= 16) ? 1 : (L > 1 && L <= 32) ? 2
              : (L > 1 && L <= WCAP) ? 3 : Q_LONG;
    }
  }
  // one queue reservation per CTA and queue: five 10-bit counts in one scan
  unsigned long long mine_q = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (qcls[j] >= 0) mine_q += 1ull << (10 * qcls[j]);
  unsigned long long tot_q = 0;
  unsigned long long pos_q = block_excl_sum64(mine_q, &tot_q, scan64);
  if (tid < 5) {
    const uint32_t cnt = (uint32_t)(tot_q >> (10 * tid)) & 1023u;
    s_qbase[tid] = cnt ? atomicAdd(&ws.st->qcount[tid], cnt) : 0u;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int qc = qcls[j];
    if (qc >= 0) {
      const uint32_t slot = s_qbase[qc] + ((uint32_t)(pos_q >> (10 * qc)) & 1023u);
      pos_q += 1ull << (10 * qc);
      // select the queue with constant indices: a run-time index into the
      // kernel-parameter struct would take a generic address of parameter space
      Frag* qp = qc == 0 ? ws.q[0] : qc == 1 ? ws.q[1] : qc == 2 ? ws.q[2] : qc == 3 ? ws.q[3] : ws.q[Q_LONG];
      qp[slot] = Frag{r0 + fstart[flo + j], flen[j]};
    }
  }
}

// ---------------------------------------------------------------------------
// K3b: queued fragments of at most WCAP bytes, several per warp, through the
// sweep engine with warp-synchronous steps only.  Lane l owns symbols
// [W_EPT*l, W_EPT*l + W_EPT) of the batch.

struct WarpEngine {
  uint32_t sym[WCAP];
  unsigned long long kr[WCAP];
  uint16_t len[WCAP];
  uint16_t ml[WCAP];
  uint16_t mr[WCAP];
  uint32_t pmin[WCAP];      // lowest rank from the fragment's first pair to this one
  uint32_t smin[WCAP];      // lowest rank from this pair to the fragment's last one
  uint8_t rs[WCAP];
  uint8_t fl[WCAP];
  uint8_t fi[WCAP];        // fragment of each symbol within the batch
  uint8_t first[W_GRAB + 1];
  long long fstart[W_GRAB];
  int foff[W_GRAB + 1];    // fragment offsets in the batch, then its size
};

__device__ __forceinline__ int warp_excl_sum(int v, int* total) {
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

__device__ __forceinline__ int warp_excl_max(int v) {
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

// Encode the batch described by W.fstart / W.foff (nfrag fragments, M symbols).
__device__ void warp_engine(WarpEngine& W, const Call& c, const Workspace& ws, const DevVocab& V, int nfrag, int M) {
  const int lane = threadIdx.x & 31;
  {
    uint32_t id[W_EPT];
#pragma unroll
    for (int r = 0; r < W_EPT; ++r) {
      const int i = lane + 32 * r;
      id[r] = 0;
      if (i < M) {
        int k = 0;
        while (k + 1 < nfrag && W.foff[k + 1] <= i) ++k;
        const int j = i - W.foff[k];
        id[r] = (uint32_t)__ldg(V.byte_id + c.text[W.fstart[k] + j]);
        W.len[i] = (uint16_t)(1u | (j == 0 ? FRAG_START : 0u));
        W.fi[i] = (uint8_t)k;
      }
    }
#pragma unroll
    for (int r = 0; r < W_EPT; ++r) {
      const int i = lane + 32 * r;
      if (i < M) {
        W.sym[i] = id[r];
        W.ml[i] = __ldg(V.max_left + id[r]);
        W.mr[i] = __ldg(V.max_right + id[r]);
      }
    }
  }
  __syncwarp();
  {
    uint32_t a[W_EPT], b[W_EPT], valid = 0;
    unsigned long long kr[W_EPT];
#pragma unroll
    for (int r = 0; r < W_EPT; ++r) {
      const int i = lane + 32 * r;
      a[r] = 0; b[r] = 0;
      if (i + 1 < M && !(W.len[i + 1] & FRAG_START)) {
        a[r] = W.sym[i];
        b[r] = W.sym[i + 1];
        valid |= 1u << r;
      }
    }
    merge_lookup_n<W_EPT>(V, a, b, valid, kr);
#pragma unroll
    for (int r = 0; r < W_EPT; ++r) {
      const int i = lane + 32 * r;
      if (i < M) W.kr[i] = ((valid >> r) & 1u) ? kr[r] : KR_WALL;
    }
  }
  __syncwarp();
  int m = M;
  for (int sweep = 0; sweep <= M; ++sweep) {
    const int lo = min(lane * W_EPT, m), hi = min(lo + W_EPT, m);
    bool anyk = false, eq = false;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = kr_rank(W.kr[i]);
      if (mergeable(k)) {
        anyk = true;
        if (i > 0 && kr_rank(W.kr[i - 1]) == k) eq = true;
      }
    }
    if (!__any_sync(0xffffffffu, anyk)) break;
    const bool runs = __any_sync(0xffffffffu, eq);
    if (runs) {
      int lastrun = -1;
      for (int i = lo; i < hi; ++i)
        if (i == 0 || kr_rank(W.kr[i - 1]) != kr_rank(W.kr[i])) lastrun = i;
      int run = warp_excl_max(lastrun);
      for (int i = lo; i < hi; ++i) {
        if (i == 0 || kr_rank(W.kr[i - 1]) != kr_rank(W.kr[i])) run = i;
        W.rs[i] = (uint8_t)run;
      }
      __syncwarp();
    }
    if (V.monotone) {
      // lowest rank over the pairs of the same fragment to the left (pmin)
      // and to the right (smin) of each pair; a wall pair is a segment of its
      // own with no rank
      uint32_t pm[W_EPT], sm[W_EPT];
      uint32_t lp = NO_RANK, lflag = 0;  // lane's suffix of prefix-min; segment restarted in lane
#pragma unroll
      for (int j = 0; j < W_EPT; ++j) {
        const int i = lo + j;
        pm[j] = NO_RANK;
        if (i < hi) {
          const uint32_t k = kr_rank(W.kr[i]);
          const bool wall = k == RANK_WALL;
          const bool start = i == 0 || wall || kr_rank(W.kr[i - 1]) == RANK_WALL;
          const uint32_t v = wall ? NO_RANK : k;
          lp = start ? v : min(lp, v);
          lflag |= start;
          pm[j] = lp;
        }
      }
      // carry from lower lanes: the prefix-min of the segment open at the lane's start
      uint32_t carry = lp, cflag = lflag;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t oc = __shfl_up_sync(0xffffffffu, carry, off);
        const uint32_t of = __shfl_up_sync(0xffffffffu, cflag, off);
        if (lane >= off) {
          if (!cflag) carry = min(carry, oc);
          cflag |= of;
        }
      }
      uint32_t in = __shfl_up_sync(0xffffffffu, carry, 1);
      if (lane == 0) in = NO_RANK;
      bool open = true;  // before the first segment start in this lane
#pragma unroll
      for (int j = 0; j < W_EPT; ++j) {
        const int i = lo + j;
        if (i < hi) {
          const uint32_t k = kr_rank(W.kr[i]);
          const bool start = i == 0 || k == RANK_WALL || kr_rank(W.kr[i - 1]) == RANK_WALL;
          if (start) open = false;
          if (open) pm[j] = min(pm[j], in);
        }
      }
      uint32_t ls = NO_RANK, rflag = 0;  // suffix-min, scanning right to left
#pragma unroll
      for (int j = W_EPT - 1; j >= 0; --j) {
        const int i = lo + j;
        sm[j] = NO_RANK;
        if (i < hi) {
          const uint32_t k = kr_rank(W.kr[i]);
          const bool wall = k == RANK_WALL;
          const bool end = i + 1 >= m || wall || kr_rank(W.kr[i + 1]) == RANK_WALL;
          const uint32_t v = wall ? NO_RANK : k;
          ls = end ? v : min(ls, v);
          rflag |= end;
          sm[j] = ls;
        }
      }
      uint32_t carry2 = ls, cflag2 = rflag;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t oc = __shfl_down_sync(0xffffffffu, carry2, off);
        const uint32_t of = __shfl_down_sync(0xffffffffu, cflag2, off);
        if (lane + off < 32) {
          if (!cflag2) carry2 = min(carry2, oc);
          cflag2 |= of;
        }
      }
      uint32_t in2 = __shfl_down_sync(0xffffffffu, carry2, 1);
      if (lane == 31) in2 = NO_RANK;
      bool open2 = true;
#pragma unroll
      for (int j = W_EPT - 1; j >= 0; --j) {
        const int i = lo + j;
        if (i < hi) {
          const uint32_t k = kr_rank(W.kr[i]);
          const bool end = i + 1 >= m || k == RANK_WALL || kr_rank(W.kr[i + 1]) == RANK_WALL;
          if (end) open2 = false;
          if (open2) sm[j] = min(sm[j], in2);
        }
      }
      // pm / sm of a pair held by another lane come through shared memory
#pragma unroll
      for (int j = 0; j < W_EPT; ++j) {
        const int i = lo + j;
        if (i < hi) { W.pmin[i] = pm[j]; W.smin[i] = sm[j]; }
      }
      __syncwarp();
      auto mlf = [&](int x) { return (int)W.ml[x]; };
      auto mrf = [&](int x) { return (int)W.mr[x]; };
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(W.kr[i]);
        bool safe = false;
        if (mergeable(k)) {
          const int u = runs ? (int)W.rs[i] : i;
          // no lower rank anywhere in the fragment beyond the direct neighbours:
          // safe without walking the length-bounded windows
          const bool left_clear = u < 2 || W.pmin[u - 2] >= k;
          const bool right_clear = i + 2 >= m || W.smin[i + 2] >= k;
          const bool nbr_ok = ((i - u) & 1) == 0 && (u == 0 || kr_rank(W.kr[u - 1]) >= k) &&
                              (i + 1 >= m || kr_rank(W.kr[i + 1]) >= k);
          if (left_clear && right_clear) safe = nbr_ok;
          else safe = pair_safe(W.len, W.kr, m, i, u, k, mlf, mrf);
        }
        W.fl[i] = safe ? 1 : 0;
      }
    } else {
      unsigned long long best = ~0ull;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = kr_rank(W.kr[i]);
        if (mergeable(k)) {
          const unsigned long long key = ((unsigned long long)k << 32) | (uint32_t)i;
          best = key < best ? key : best;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o < best ? o : best;
      }
      for (int i = lo; i < hi; ++i) W.fl[i] = ((uint32_t)best == (uint32_t)i) ? 1 : 0;
    }
    __syncwarp();
    // merge, look up the new pairs, compact (through registers)
    uint32_t nsym[W_EPT];
    uint16_t nlen[W_EPT], nml[W_EPT], nmr[W_EPT];
    uint8_t nfi[W_EPT];
    unsigned long long nkr[W_EPT];
    uint32_t keep = 0;
    uint32_t la[W_EPT], lb[W_EPT], need = 0, merged = 0;
#pragma unroll
    for (int j = 0; j < W_EPT; ++j) {
      const int i = lo + j;
      nsym[j] = 0; nlen[j] = 0; nml[j] = 0; nmr[j] = 0; nfi[j] = 0; nkr[j] = KR_WALL; la[j] = 0; lb[j] = 0;
      if (i < hi && !(i > 0 && W.fl[i - 1])) {
        keep |= 1u << j;
        const bool mg = W.fl[i] != 0;
        if (mg) {
          merged |= 1u << j;
          nsym[j] = kr_result(W.kr[i]);
          nlen[j] = (uint16_t)(((W.len[i] & LEN_MASK) + (W.len[i + 1] & LEN_MASK)) | (W.len[i] & FRAG_START));
        } else {
          nsym[j] = W.sym[i];
          nlen[j] = W.len[i];
          nml[j] = W.ml[i];
          nmr[j] = W.mr[i];
        }
        nfi[j] = W.fi[i];
        const int jn = mg ? i + 2 : i + 1;  // the next symbol that survives
        if (jn >= m || (W.len[jn] & FRAG_START)) {
          nkr[j] = KR_WALL;
        } else if (!mg && !W.fl[jn]) {
          nkr[j] = W.kr[i];  // an unchanged pair keeps its key
        } else {
          la[j] = nsym[j];
          lb[j] = W.fl[jn] ? kr_result(W.kr[jn]) : W.sym[jn];
          need |= 1u << j;
        }
      }
    }
    // operand bounds of new symbols and keys of new pairs, loads overlapped
#pragma unroll
    for (int j = 0; j < W_EPT; ++j)
      if ((merged >> j) & 1u) { nml[j] = __ldg(V.max_left + nsym[j]); nmr[j] = __ldg(V.max_right + nsym[j]); }
    {
      unsigned long long got[W_EPT];
      merge_lookup_n<W_EPT>(V, la, lb, need, got);
#pragma unroll
      for (int j = 0; j < W_EPT; ++j)
        if ((need >> j) & 1u) nkr[j] = got[j];
    }
    int newm = 0;
    const int base = warp_excl_sum(__popc(keep), &newm);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < W_EPT; ++j) {
      if ((keep >> j) & 1u) {
        const int p = base + __popc(keep & ((1u << j) - 1u));
        W.sym[p] = nsym[j];
        W.len[p] = nlen[j];
        W.kr[p] = nkr[j];
        W.ml[p] = nml[j];
        W.mr[p] = nmr[j];
        W.fi[p] = nfi[j];
      }
    }
    m = newm;
    __syncwarp();
    if (sweep == M && lane == 0) atomicExch(&ws.st->code, ST_EINTERNAL);  // cannot happen: every sweep merges
  }
  // ids at each fragment's byte offset, and their number
  for (int i = lane; i < m; i += 32)
    if (W.len[i] & FRAG_START) W.first[W.fi[i]] = (uint8_t)i;
  if (lane == 0) W.first[nfrag] = (uint8_t)m;
  __syncwarp();
  for (int i = lane; i < m; i += 32) {
    const int k = W.fi[i];
    ws.tok[W.fstart[k] + (i - W.first[k])] = (int32_t)W.sym[i];
  }
  if (lane < nfrag) ws.fcnt[W.fstart[lane]] = W.first[lane + 1] - W.first[lane];
  __syncwarp();
}

// Segment engine: fragments of at most W bytes (W in {8, 16, 32}), one symbol
// per lane, 32 / W fragments per warp, each in its own W-lane segment.  The
// same sweep as the warp engine (every certified-safe pair merges), with all
// neighbour access through segment-local shuffles.
template <int W>
__device__ void segment_engine(const Call& c, const Workspace& ws, const DevVocab& V, long long a, int len) {
  const int lane = threadIdx.x & 31;
  const int i = lane & (W - 1);              // position in the segment
  const int seg0 = lane & ~(W - 1);          // first lane of the segment
  const uint32_t segbits = (W == 32 ? 0xffffffffu : ((1u << W) - 1u)) << seg0;
  int m = len;                               // symbols in this segment (0: no fragment)
  uint32_t sym = 0, mlv = 0, mrv = 0, lenb = 0;
  if (i < m) {
    const int32_t id = __ldg(V.byte_id + c.text[a + i]);
    sym = (uint32_t)id;
    mlv = __ldg(V.max_left + id);
    mrv = __ldg(V.max_right + id);
    lenb = 1;
  }
  unsigned long long kr = KR_WALL;
  {
    const uint32_t nxt = __shfl_down_sync(0xffffffffu, sym, 1, W);
    uint32_t p[1] = {sym}, q[1] = {nxt};
    unsigned long long got[1];
    merge_lookup_n<1>(V, p, q, (i + 1 < m) ? 1u : 0u, got);
    if (i + 1 < m) kr = got[0];
  }
  for (int sweep = 0; sweep <= W; ++sweep) {
    const uint32_t k = kr_rank(kr);
    const bool mrg = i + 1 < m && mergeable(k);
    if (!__any_sync(0xffffffffu, mrg)) break;
    // ranks of the neighbouring pairs
    const uint32_t kl = __shfl_up_sync(0xffffffffu, k, 1, W);
    const uint32_t kn = __shfl_down_sync(0xffffffffu, k, 1, W);
    // run start of equal-rank pairs (runs of one symbol x with merge (x,x))
    int u = i;
    const bool eq = mrg && i > 0 && kl == k;
    if (__any_sync(0xffffffffu, eq)) {
      int st = (i + 1 < m && !(i > 0 && kl == k)) ? i : -1;
#pragma unroll
      for (int off = 1; off < W; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, st, off, W);
        if (i >= off) st = max(st, o);
      }
      u = st < 0 ? i : st;
    }
    // lowest rank over pairs [0, x] (pm) and [x, m-2] (sm) of the fragment
    const uint32_t kv = (i + 1 < m) ? k : NO_RANK;
    uint32_t pm = kv, sm = kv;
#pragma unroll
    for (int off = 1; off < W; off <<= 1) {
      const uint32_t o1 = __shfl_up_sync(0xffffffffu, pm, off, W);
      const uint32_t o2 = __shfl_down_sync(0xffffffffu, sm, off, W);
      if (i >= off) pm = min(pm, o1);
      if (i + off < W) sm = min(sm, o2);
    }
    const uint32_t pm_u2 = __shfl_sync(0xffffffffu, pm, seg0 + max(u - 2, 0));
    const uint32_t kl_u = __shfl_sync(0xffffffffu, k, seg0 + max(u - 1, 0));
    const uint32_t sm_i2 = __shfl_down_sync(0xffffffffu, sm, 2, W);
    const uint32_t ml_u = __shfl_sync(0xffffffffu, mlv, seg0 + u);
    const uint32_t mr_i1 = __shfl_down_sync(0xffffffffu, mrv, 1, W);
    bool safe = false;
    bool need_scan = false;
    if (mrg) {
      const bool nbr_ok = ((i - u) & 1) == 0 && (u == 0 || kl_u >= k) && (i + 2 >= m || kn >= k);
      const bool left_clear = u < 2 || pm_u2 >= k;
      const bool right_clear = i + 3 >= m || sm_i2 >= k;
      safe = nbr_ok && left_clear && right_clear;
      need_scan = nbr_ok && !(left_clear && right_clear);
    }
    // exact length-bounded windows where a lower rank exists further away
    if (__any_sync(0xffffffffu, need_scan)) {
      bool ok = need_scan;
      // left: initiator pair q <= u-2 grows a token ending at u-1
      int cum = __shfl_sync(0xffffffffu, (int)lenb, seg0 + max(u - 1, 0));
      bool done = !(need_scan && u >= 2);
      for (int step = 2; step < W; ++step) {
        const int q = u - step;
        const int qq = max(q, 0);
        const uint32_t kq = __shfl_sync(0xffffffffu, k, seg0 + qq);
        const int lq = __shfl_sync(0xffffffffu, (int)lenb, seg0 + qq);
        if (!done) {
          if (q < 0) done = true;
          else {
            cum += lq;
            if (cum > (int)ml_u) done = true;
            else if (kq < k) { ok = false; done = true; }
          }
        }
        if (!__any_sync(0xffffffffu, !done)) break;
      }
      // right: initiator pair q >= i+2 grows a token starting at i+2
      cum = __shfl_sync(0xffffffffu, (int)lenb, seg0 + min(i + 2, W - 1));
      done = !(need_scan && ok && i + 3 < m);
      for (int step = 2; step < W; ++step) {
        const int q = i + step;
        const int qq = min(q, W - 1);
        const uint32_t kq = __shfl_sync(0xffffffffu, k, seg0 + qq);
        const int lq = __shfl_sync(0xffffffffu, (int)lenb, seg0 + min(q + 1, W - 1));
        if (!done) {
          if (q >= m - 1) done = true;
          else {
            cum += lq;
            if (cum > (int)mr_i1) done = true;
            else if (kq < k) { ok = false; done = true; }
          }
        }
        if (!__any_sync(0xffffffffu, !done)) break;
      }
      if (need_scan) safe = ok;
    }
    if (!V.monotone) {
      // the rule itself: only the leftmost minimum pair of each fragment
      uint32_t best = mrg ? k : NO_RANK;
      int bi = i;
#pragma unroll
      for (int off = W / 2; off > 0; off >>= 1) {
        const uint32_t ob = __shfl_xor_sync(0xffffffffu, best, off, W);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off, W);
        if (ob < best || (ob == best && oi < bi)) { best = ob; bi = oi; }
      }
      safe = mrg && bi == i;
    }
    // merge: a safe pair's left symbol takes the result, its right one goes
    const bool dead = __shfl_up_sync(0xffffffffu, safe ? 1 : 0, 1, W) != 0 && i > 0;
    const uint32_t nlen = lenb + (safe ? (uint32_t)__shfl_down_sync(0xffffffffu, (int)lenb, 1, W) : 0u);
    uint32_t nsym = safe ? kr_result(kr) : sym;
    const bool keep = i < m && !dead;
    const uint32_t km = (__ballot_sync(0xffffffffu, keep) & segbits) >> seg0;
    const bool chg = safe;
    const int newm = __popc(km);
    // compaction: new position p takes the (p+1)-th survivor
    const int src = i < newm ? (int)__fns(km, 0, i + 1) : i;
    nsym = __shfl_sync(0xffffffffu, nsym, seg0 + src);
    const uint32_t nl2 = __shfl_sync(0xffffffffu, nlen, seg0 + src);
    const bool c2 = __shfl_sync(0xffffffffu, chg ? 1 : 0, seg0 + src) != 0;
    const unsigned long long okr = __shfl_sync(0xffffffffu, kr, seg0 + src);
    uint32_t nml = __shfl_sync(0xffffffffu, mlv, seg0 + src);
    uint32_t nmr = __shfl_sync(0xffffffffu, mrv, seg0 + src);
    m = newm;
    sym = i < m ? nsym : 0u;
    lenb = i < m ? nl2 : 0u;
    if (i < m && c2) { nml = __ldg(V.max_left + sym); nmr = __ldg(V.max_right + sym); }
    mlv = nml;
    mrv = nmr;
    // keys: unchanged pairs keep theirs, pairs touching a new symbol are looked up
    const bool c_next = __shfl_down_sync(0xffffffffu, c2 ? 1 : 0, 1, W) != 0;
    const uint32_t nxt = __shfl_down_sync(0xffffffffu, sym, 1, W);
    const bool look = i + 1 < m && (c2 || c_next);
    uint32_t p[1] = {sym}, q[1] = {nxt};
    unsigned long long got[1];
    merge_lookup_n<1>(V, p, q, look ? 1u : 0u, got);
    kr = (i + 1 < m) ? (look ? got[0] : okr) : KR_WALL;
    if (sweep == W && i == 0 && m > 1) atomicExch(&ws.st->code, ST_EINTERNAL);
  }
  if (i < m) ws.tok[a + i] = (int32_t)sym;
  if (i == 0 && len > 0) ws.fcnt[a] = m;
}

template <int W>
__device__ void drain_segment_queue(const Call& c, const Workspace& ws, const DevVocab& V, const Frag* queue,
                                    const uint32_t* qcount, uint32_t* qtaken) {
  constexpr int PER = 32 / W;  // fragments per warp
  const int lane = threadIdx.x & 31;
  const uint32_t count = *(volatile const uint32_t*)qcount;
  while (true) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(qtaken, (uint32_t)PER);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (base >= count) break;
    const uint32_t k = base + (uint32_t)(lane / W);
    Frag f{0, 0};
    if (k < count) f = queue[k];
    segment_engine<W>(c, ws, V, f.start, (int)f.len);
  }
}

__global__ void __launch_bounds__(W_WARPS * 32, 4) k_bpe_warp(Call c, Workspace ws, DevVocab V) {
  __shared__ WarpEngine engines[W_WARPS];
  WarpEngine& W = engines[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const uint32_t count = *(volatile uint32_t*)&ws.st->qcount[3];
  // longest fragments first: warp engine (33..128 bytes), then segments of 32, 16, 8
  while (true) {
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&ws.st->qtaken[3], (uint32_t)W_GRAB);
    base = __shfl_sync(0xffffffffu, base, 0);
    if (base >= count) break;
    const int ng = (int)min((uint32_t)W_GRAB, count - base);
    Frag f{0, 0};
    if (lane < ng) f = ws.q[3][base + lane];
    // batches of consecutive entries with at most WCAP symbols
    for (int k0 = 0; k0 < ng;) {
      const int l = (lane >= k0 && lane < ng) ? (int)f.len : 0;
      int tot = 0;
      const int ex = warp_excl_sum(l, &tot);
      const bool fits = lane >= k0 && lane < ng && ex + l <= WCAP;
      const uint32_t mask = __ballot_sync(0xffffffffu, fits);
      const int k1 = k0 + __popc(mask);
      if (fits) {
        W.fstart[lane - k0] = f.start;
        W.foff[lane - k0] = ex;
      }
      const int M = __shfl_sync(0xffffffffu, ex + l, k1 - 1);
      if (lane == 0) W.foff[k1 - k0] = M;
      __syncwarp();
      warp_engine(W, c, ws, V, k1 - k0, M);
      k0 = k1;
    }
  }
  drain_segment_queue<32>(c, ws, V, ws.q[2], &ws.st->qcount[2], &ws.st->qtaken[2]);
  drain_segment_queue<16>(c, ws, V, ws.q[1], &ws.st->qcount[1], &ws.st->qtaken[1]);
  drain_segment_queue<8>(c, ws, V, ws.q[0], &ws.st->qcount[0], &ws.st->qtaken[0]);
}

// ---------------------------------------------------------------------------
// K4: fragments longer than a warp batch holds, one CTA each, in global
// memory at the fragment's byte offsets (double-buffered)

__global__ void __launch_bounds__(LONG_THREADS) k_bpe_long(Call c, Workspace ws, DevVocab V) {
  __shared__ int sh[LONG_THREADS / 32];
  __shared__ unsigned long long sh64[LONG_THREADS / 32];
  __shared__ uint32_t s_idx;
  __shared__ unsigned long long s_end;
  const int tid = threadIdx.x, T = blockDim.x;
  const uint32_t count = *(volatile uint32_t*)&ws.st->qcount[Q_LONG];
  while (true) {
    if (tid == 0) s_idx = atomicAdd(&ws.st->qtaken[Q_LONG], 1u);
    __syncthreads();
    const uint32_t idx = s_idx;
    __syncthreads();
    if (idx >= count) break;
    const Frag f = ws.q[Q_LONG][idx];
    // end: known from the queue entry, or the next fragment start after
    // f.start (or the text end)
    if (tid == 0) s_end = f.len > 0 ? (unsigned long long)(f.start + f.len) : (unsigned long long)c.n;
    __syncthreads();
    const long long w0 = (f.start + 1) >> 5, wn = f.len > 0 ? w0 : (c.n + 31) >> 5;
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
    if (tid == 0) ws.fcnt[a] = m;
    __syncthreads();
  }
}

void launch_settle(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s) {
  k_settle<<<(unsigned)n_bchunks(c.n), B_THREADS, 0, s>>>(c, w, v);
}

void launch_bpe_warp(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_warp<<<n_sms * 4, W_WARPS * 32, 0, s>>>(c, w, v);
}

void launch_bpe_long(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s) {
  k_bpe_long<<<n_sms, LONG_THREADS, 0, s>>>(c, w, v);
}

}  // namespace tokgb
