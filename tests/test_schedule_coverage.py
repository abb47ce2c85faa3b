"""CPU test of the kernels' work decomposition.  A host program built with
nvcc walks every forward (and dQ) work item -- rank r's rank-local query tile
t -- and every dK/dV work item -- key tile jk of chunk c -- with the same
__host__ __device__ geometry functions the kernels use (fwd_tile_qmax,
fwd_chunk_tiles, ring_src/ring_chunk, bwd_kv_range, bwd_q_tile_visits and the
planner's cost functions), on random ragged metadata.  The checks here derive
positions from the chunking reading alone (rank r holds chunks r and
2cp-1-r; chunk = padded length / 2cp): every (query, key) pair the mask
allows is visited exactly once, no visited tile is useless, the walk follows
ring order, and the planner's cost equals the tiles walked."""

import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "packed_sequence_context_gb300", "csrc")
TILE = 128

WALKER = r"""
#include <cstdio>
#include "common.cuh"
using namespace thd;

int main() {
  int ncase;
  if (scanf("%d", &ncase) != 1) return 1;
  for (int k = 0; k < ncase; ++k) {
    int B, cp, causal;
    if (scanf("%d %d %d", &B, &cp, &causal) != 3) return 1;
    printf("C %d\n", k);
    for (int b = 0; b < B; ++b) {
      int Lq, Pq, Lkv, Pkv;
      if (scanf("%d %d %d %d", &Lq, &Pq, &Lkv, &Pkv) != 4) return 1;
      SeqGeom g;
      g.q_off = 0;
      g.kv_off = 0;
      g.Lq = Lq;
      g.Lkv = Lkv;
      g.cbq = Pq / (2 * cp);
      g.cbkv = Pkv / (2 * cp);
      g.koff = causal == 2 ? Lkv - Lq : 0;   // bottom-right: j <= i + Lkv - Lq
      for (int r = 0; r < cp; ++r)
        for (int t = 0; t < ceil_div(2 * g.cbq, kTile); ++t) {
          const int qmax = fwd_tile_qmax(g, r, t, cp);
          printf("F %d %d %d %d %d", b, r, t, qmax, fwd_item_tiles(g, r, t, cp, causal != 0, 0, cp));
          for (int i = 0; i < cp; ++i) {
            const int s = ring_src(r, i, cp);
            for (int e = 0; e < 2; ++e) {
              const int c = ring_chunk(s, e, cp);
              const int n = fwd_chunk_tiles(g, c, qmax, causal != 0);
              for (int j = 0; j < n; ++j) printf(" %d:%d", c, j);
            }
          }
          printf("\n");
        }
      for (int c = 0; c < 2 * cp; ++c)
        for (int jk = 0; jk < ceil_div(g.cbkv, kTile); ++jk) {
          int kf, kl;
          bwd_kv_range(g, c, jk, kf, kl);
          printf("K %d %d %d %d %d %d", b, c, jk, kf, kl, bwd_item_qtiles(g, c, jk, cp, causal != 0));
          if (kf <= kl) {
            const int s = chunk_owner(c, cp);
            const int nq = ceil_div(g.cbq, kTile);
            for (int i = 0; i < cp; ++i) {
              const int r = (s + i) % cp;
              for (int e = 0; e < 2; ++e) {
                const int qc = e == 0 ? r : 2 * cp - 1 - r;
                for (int jq = 0; jq < nq; ++jq)
                  if (bwd_q_tile_visits(g, qc, jq, kf, kl, causal != 0)) printf(" %d:%d", qc, jq);
              }
            }
          }
          printf("\n");
        }
    }
  }
  return 0;
}
"""


def _cases(seed=0, n=40):
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        cp = int(rng.choice([1, 2, 3, 4, 8]))
        causal = (1, 1, 2, 0)[k % 4]   # top-left, bottom-right (Lq != Lkv), none
        B = int(rng.integers(1, 5))
        seqs = []
        for _ in range(B):
            unit = 2 * cp
            Pq = unit * int(rng.integers(0, 1200 // unit + 1))
            Lq = int(rng.integers(0, Pq + 1)) if rng.random() < 0.5 else Pq
            if causal == 1:
                Pkv, Lkv = Pq, Lq
            else:
                Pkv = unit * int(rng.integers(0, 900 // unit + 1))
                Lkv = int(rng.integers(0, Pkv + 1))
            seqs.append((Lq, Pq, Lkv, Pkv))
        out.append((cp, causal, seqs))
    # fixed edge cases: exact tile multiples, one-row chunks, a long single sequence
    out.append((4, 1, [(1024, 1024, 1024, 1024)]))
    out.append((8, 1, [(16, 16, 16, 16), (0, 32, 0, 32)]))
    out.append((1, 1, [(1000, 1024, 1000, 1024)]))
    out.append((2, 0, [(260, 264, 5, 8)]))
    # bottom-right: fewer queries than keys, more queries than keys (the first Lq - Lkv see nothing)
    out.append((4, 2, [(100, 128, 1000, 1024), (1000, 1024, 100, 128), (0, 8, 40, 48)]))
    return out


@pytest.fixture(scope="module")
def walker(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("walker")
    src = d / "walker.cu"
    src.write_text(WALKER)
    exe = d / "walker"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _pos(p, r, cb, cp):
    """Sequence position of rank r's rank-local row p (chunk r, then chunk 2cp-1-r)."""
    return r * cb + p if p < cb else (2 * cp - 1 - r) * cb + (p - cb)


def _sees(i, j, Lkv, causal, koff=0):
    return j < Lkv and (j <= i + koff if causal else True)


def test_every_allowed_pair_is_visited_exactly_once(walker):
    cases = _cases()
    inp = [str(len(cases))]
    for cp, causal, seqs in cases:
        inp.append(f"{len(seqs)} {cp} {causal}")
        inp += [" ".join(map(str, s)) for s in seqs]
    r = subprocess.run([str(walker)], input="\n".join(inp) + "\n", capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    blocks = r.stdout.split("C ")[1:]
    assert len(blocks) == len(cases)
    for (cp, causal, seqs), block in zip(cases, blocks):
        lines = block.strip().split("\n")[1:]
        fwd = [ln.split() for ln in lines if ln.startswith("F")]
        bwd = [ln.split() for ln in lines if ln.startswith("K")]
        for b, (Lq, Pq, Lkv, Pkv) in enumerate(seqs):
            cbq, cbkv = Pq // (2 * cp), Pkv // (2 * cp)
            koff = Lkv - Lq if causal == 2 else 0

            def key_range(c, j):
                lo = c * cbkv + j * TILE
                return lo, min(c * cbkv + min((j + 1) * TILE, cbkv), Lkv)   # [lo, hi)

            # ---- forward / dQ items: rank r, rank-local query tile t
            items = [f for f in fwd if int(f[1]) == b]
            assert len(items) == cp * -(-2 * cbq // TILE)
            for f in items:
                r, t, qmax, cost = int(f[2]), int(f[3]), int(f[4]), int(f[5])
                tiles = [tuple(map(int, x.split(":"))) for x in f[6:]]
                rows = [_pos(p, r, cbq, cp) for p in range(t * TILE, min(t * TILE + TILE, 2 * cbq))]
                valid = [i for i in rows if i < Lq]
                assert qmax == (max(valid) if valid else -1)
                assert cost == len(tiles)
                # ring order: step i holds rank (r - i) mod cp, chunks s then 2cp-1-s, tiles in order
                order = [c for i in range(cp) for c in ((r - i) % cp, 2 * cp - 1 - (r - i) % cp)]
                assert [c for c, _ in tiles] == sorted((c for c, _ in tiles), key=order.index)
                for c in set(c for c, _ in tiles):
                    js = [j for cc, j in tiles if cc == c]
                    assert js == list(range(len(js)))
                # every row's visible keys are a prefix: all of [0, need_hi] must be covered, once
                need_hi = (min(qmax + koff, Lkv - 1) if causal else Lkv - 1) if valid else -1
                covered = set()
                for c, j in tiles:
                    lo, hi = key_range(c, j)
                    assert lo < hi, "a visited key tile holds no valid key"
                    assert lo <= need_hi, "a visited key tile no query of the tile sees"
                    assert covered.isdisjoint(range(lo, hi))
                    covered.update(range(lo, hi))
                assert covered >= set(range(need_hi + 1)), (b, r, t)
            # ---- dK/dV items: key tile jk of chunk c
            kitems = [k for k in bwd if int(k[1]) == b]
            assert len(kitems) == 2 * cp * -(-cbkv // TILE)
            seen_keys = []
            for k in kitems:
                c, jk, kf, kl, cost = (int(x) for x in k[2:7])
                qtiles = [tuple(map(int, x.split(":"))) for x in k[7:]]
                lo, hi = key_range(c, jk)
                if lo < hi:
                    assert (kf, kl) == (lo, hi - 1)
                else:
                    assert kf > kl
                assert cost == len(qtiles)
                if kf > kl:
                    assert not qtiles
                    continue
                seen_keys += list(range(kf, kl + 1))
                s = c if c < cp else 2 * cp - 1 - c
                order = [qc for i in range(cp) for qc in ((s + i) % cp, 2 * cp - 1 - (s + i) % cp)]
                assert [qc for qc, _ in qtiles] == sorted((qc for qc, _ in qtiles), key=order.index)
                # the queries that see some key of [kf, kl]: i + koff >= kf under a causal mask, all otherwise
                need = set(range(max(kf - koff, 0) if causal else 0, Lq))
                rows_in = set()
                for qc, jq in qtiles:
                    q_lo, q_hi = qc * cbq + jq * TILE, min(qc * cbq + min((jq + 1) * TILE, cbq), Lq)
                    assert not need.isdisjoint(range(q_lo, q_hi)), "a visited query tile no query of which sees the keys"
                    assert rows_in.isdisjoint(range(q_lo, q_hi))
                    rows_in.update(range(q_lo, q_hi))
                assert rows_in >= need, (b, c, jk)
            assert sorted(seen_keys) == list(range(Lkv))
