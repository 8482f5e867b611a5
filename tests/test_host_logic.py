"""The library's host-side scheduling logic, compiled from its own sources and run
on the CPU (no GPU involved): the split plan's partition of the global page list
over the persistent workers, the split slots the attend kernels write and the
merge kernels read, the decode workspace layout (with the plan block's
sections), the no-allocation decode's worker count, the producer's choice of K
split and its workspace size, and the query layout of several query tokens per
row."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mla_absorbed_latent_gb300", "csrc")

HARNESS = r"""
#include "cache_project.cu"
#include "tensor_map.cu"
#include <cstdio>
#include <vector>
using namespace mla;

static int fails = 0;
#define CHECK(cond, ...)                                   \
  do {                                                     \
    if (!(cond)) {                                         \
      if (++fails <= 20) {                                 \
        std::printf("FAIL %s: ", #cond);                   \
        std::printf(__VA_ARGS__);                          \
        std::printf("\n");                                 \
      }                                                    \
    }                                                      \
  } while (0)

int main() {
  // 1. T tiles cut into W contiguous ranges: ranges cover [0, T) in order and
  //    worker_of_tile names the range that holds each tile
  for (long long T = 1; T <= 700; T += (T < 100 ? 1 : 37))
    for (long long W = 1; W <= 320; W += (W < 40 ? 1 : 13)) {
      CHECK(worker_begin(0, T, W) == 0, "T=%lld W=%lld", T, W);
      CHECK(worker_begin(W, T, W) == T, "T=%lld W=%lld", T, W);
      for (long long w = 0; w < W; ++w)
        CHECK(worker_begin(w, T, W) <= worker_begin(w + 1, T, W), "T=%lld W=%lld w=%lld", T, W, w);
      for (long long x = 0; x < T; ++x) {
        const int w = worker_of_tile(x, T, W);
        CHECK(w >= 0 && w < W && worker_begin(w, T, W) <= x && x < worker_begin(w + 1, T, W),
              "T=%lld W=%lld x=%lld w=%d", T, W, x, w);
      }
    }

  // 1b. the split slots: a worker writes its split of row b to slot w + b; the
  //     merge reads row b's slots [worker_of_tile(first tile) + b,
  //     worker_of_tile(last tile) + b] and a row group's CTA loads the slots
  //     [s_lo, s_hi) of its rows.  Over ragged rows (empty ones included):
  //     written slots are distinct and below W + B, each slot a row reads was
  //     written for that row or belongs to a worker without tiles (weight 0),
  //     and a group's window holds every slot its rows read
  {
    unsigned rng = 777u;
    auto rnd = [&](unsigned m) { rng = rng * 1103515245u + 12345u; return (rng >> 8) % m; };
    const int gBs[] = {1, 2, 5, 33, 64, 130, 300}, gWs[] = {1, 2, 7, 76, 152}, RBs[] = {16, 32, 64};
    for (int B : gBs)
      for (int W : gWs)
        for (int trial = 0; trial < 4; ++trial) {
          std::vector<long long> pre(B + 1, 0);
          for (int b = 0; b < B; ++b) {
            const unsigned k = rnd(10);
            pre[b + 1] = pre[b] + (k < 2 ? 0 : k < 6 ? (long long)rnd(3) + 1 : (long long)rnd(300) + 1);
          }
          const long long T = pre[B];
          if (T == 0) continue;
          std::vector<int> owner(W + B, -1);  // row whose split a slot holds
          for (int w = 0; w < W; ++w) {
            const long long a0 = worker_begin(w, T, W), a1 = worker_begin(w + 1, T, W);
            for (int b = 0; b < B; ++b)
              if (pre[b] < a1 && pre[b + 1] > a0) {
                const int s = w + b;
                CHECK(s < W + B && owner[s] < 0, "B=%d W=%d w=%d b=%d: slot %d", B, W, w, b, s);
                if (s < W + B) owner[s] = b;
              }
          }
          std::vector<int> rx(B, 1), ry(B, 0);
          for (int b = 0; b < B; ++b) {
            if (pre[b + 1] == pre[b]) continue;
            rx[b] = worker_of_tile(pre[b], T, W) + b;
            ry[b] = worker_of_tile(pre[b + 1] - 1, T, W) + b;
            for (int s = rx[b]; s <= ry[b]; ++s) {
              const long long w = s - b;
              const bool empty = worker_begin(w, T, W) == worker_begin(w + 1, T, W);
              CHECK(s >= 0 && s < W + B && (owner[s] == b || (empty && owner[s] < 0)), "B=%d W=%d b=%d s=%d", B, W,
                    b, s);
            }
            for (int s = 0; s < W + B; ++s)
              if (owner[s] == b) CHECK(rx[b] <= s && s <= ry[b], "B=%d W=%d b=%d: slot %d unread", B, W, b, s);
          }
          for (int RB : RBs)
            for (int b0 = 0; b0 < B; b0 += RB) {
              const int b_end = b0 + RB < B ? b0 + RB : B;
              const long long t0 = pre[b0], t1 = pre[b_end];
              if (t1 <= t0) continue;
              const int s_lo = worker_of_tile(t0, T, W) + b0, s_hi = worker_of_tile(t1 - 1, T, W) + b_end;
              CHECK(s_lo >= 0 && s_hi <= W + B, "B=%d W=%d b0=%d: [%d, %d)", B, W, b0, s_lo, s_hi);
              for (int b = b0; b < b_end; ++b)
                if (rx[b] <= ry[b]) CHECK(s_lo <= rx[b] && ry[b] < s_hi, "B=%d W=%d RB=%d b=%d", B, W, RB, b);
            }
        }
  }

  // 2. decode workspace: regions in order, 1 KB aligned, each large enough
  const int Bs[] = {1, 7, 64, 128, 1000}, Hs[] = {16, 128}, Ws[] = {1, 152, 304};
  for (int B : Bs)
    for (int H : Hs)
      for (int Wk : Ws) {
        const WsLayout L = ws_layout(B, H, Wk);
        CHECK(L.q_cat == 0, "B=%d", B);
        CHECK(L.plan >= L.q_cat + (size_t)B * H * DK * 2, "B=%d H=%d", B, H);
        CHECK(L.part_o >= L.plan + (size_t)(PLAN_HDR + 3 * B + 1 + Wk) * 4, "B=%d W=%d", B, Wk);
        CHECK(plan_off_seq(B) == PLAN_HDR + B + 1 && plan_off_fix(B) == plan_off_seq(B) + B &&
                  plan_off_wrow(B) == plan_off_fix(B) + B && PLAN_CTX * 4 + sizeof(FixCtx) <= PLAN_HDR * 4,
              "B=%d", B);
        CHECK(L.part_lse >= L.part_o + (size_t)(Wk + B) * H * DC * 2, "B=%d H=%d W=%d", B, H, Wk);
        CHECK(L.total >= L.part_lse + (size_t)(Wk + B) * H * 4, "B=%d H=%d W=%d", B, H, Wk);
        CHECK(L.plan % 1024 == 0 && L.part_o % 1024 == 0 && L.part_lse % 1024 == 0 && L.total % 1024 == 0,
              "B=%d H=%d W=%d", B, H, Wk);
        CHECK(L.max_segments == Wk + B, "B=%d W=%d", B, Wk);
      }

  // 3. the producer's K split: within [1, hidden/64], forced values honoured (capped),
  //    automatic ones only when the tiles leave SMs idle, every split non-empty,
  //    and a workspace exactly when there is a split
  const long long ntoks[] = {1, 64, 127, 128, 129, 1000, 9728, 9729, 32768};
  const int hiddens[] = {64, 128, 2048, 7168, 65536}, smss[] = {1, 2, 148, 152}, reqs[] = {0, 1, 3, 5, 1000};
  for (long long ntok : ntoks)
    for (int hidden : hiddens)
      for (int sms : smss)
        for (int req : reqs) {
          const int k = project_splits(ntok, hidden, sms, req);
          const int chunks = hidden / 64;
          const long long mtiles = (ntok + 127) / 128;
          CHECK(k >= 1 && k <= chunks, "ntok=%lld hidden=%d sms=%d req=%d k=%d", ntok, hidden, sms, req, k);
          if (req > 0) {
            CHECK(k == (req < chunks ? req : chunks), "req=%d chunks=%d k=%d", req, chunks, k);
          } else if (2 * mtiles >= sms) {
            CHECK(k == 1, "ntok=%lld sms=%d k=%d", ntok, sms, k);
          } else {
            const long long cap = chunks / 2 > 1 ? chunks / 2 : 1;  // at least two 64-wide chunks per pair
            const long long want = sms / (2 * mtiles);
            CHECK(k <= cap && k <= (want > 1 ? want : 1), "ntok=%lld hidden=%d sms=%d k=%d", ntok, hidden, sms, k);
          }
          for (int s = 0; s < k; ++s)
            CHECK((long long)(s + 1) * chunks / k - (long long)s * chunks / k >= 1, "chunks=%d k=%d s=%d", chunks, k,
                  s);
          const size_t ws = project_workspace_bytes(ntok, k);
          if (k == 1) {
            CHECK(ws == 0, "ntok=%lld", ntok);
          } else {
            // one fp32 partial payload per (pair, token)
            CHECK(ws >= (size_t)k * ntok * DK * 4 && ws % 256 == 0, "ntok=%lld k=%d", ntok, k);
          }
        }
  // 3b. the few-token producer (at most 64 tokens): slices of the hidden
  //     dimension within [1, hidden/64], at most 8 chunks of 64 each, about one
  //     CTA per SM when the hidden dimension allows it, and one fp32 partial
  //     payload per slice and token
  for (int hidden : hiddens)
    for (int sms : smss) {
      const int k = project_small_splits(hidden, sms);
      const int chunks = hidden / 64;
      CHECK(k >= 1 && k <= chunks && (chunks + k - 1) / k <= 8, "hidden=%d sms=%d k=%d", hidden, sms, k);
      CHECK(k >= (sms / 9 < chunks ? sms / 9 : chunks), "hidden=%d sms=%d k=%d", hidden, sms, k);
      for (long long ntok = 1; ntok <= PROJECT_SMALL_TOKENS; ntok += 21) {
        const size_t ws = project_small_workspace_bytes(ntok, k);
        CHECK(ws >= (size_t)k * ntok * DK * 4 && ws % 256 == 0, "ntok=%lld k=%d", ntok, k);
      }
    }
  // 4. the no-allocation decode's worker count: the largest count <= want whose
  //    workspace fits the capacity, 0 when one worker does not fit
  const size_t caps[] = {1u << 20, 16u << 20, 64ull << 20};
  const int wants[] = {1, 76, 304};
  for (size_t cap : caps)
    for (int H : Hs)
      for (int want : wants)
        for (int B = 1; B <= 2000; B += (B < 300 ? 7 : 101)) {
          const int w = fitting_workers(B, H, want, cap);
          CHECK(w >= 0 && w <= want, "B=%d H=%d want=%d w=%d", B, H, want, w);
          if (w > 0) {
            CHECK(ws_layout(B, H, w).total <= cap, "B=%d H=%d w=%d", B, H, w);
            if (w < want) CHECK(ws_layout(B, H, w + 1).total > cap, "B=%d H=%d w=%d", B, H, w);
          } else {
            CHECK(ws_layout(B, H, 1).total > cap, "B=%d H=%d", B, H);
          }
        }
  // 5. the query layout of several query tokens per row (G = 128 / H tokens of
  //    a row per virtual row of 128 MMA rows, NG virtual rows per row): every
  //    (row, token, head) is one virtual head of one virtual row, whose flat
  //    query row is that token's, and whose causal shift is the number of its
  //    virtual row's view tokens after its own position; padding lanes see
  //    nothing
  {
    const int qHs[] = {16, 128}, qTs[] = {1, 2, 3, 8, 9, 25, 64};
    for (int H : qHs)
      for (int T : qTs) {
        const int G = 128 / H;
        const QSpec qs{T, G, (T + G - 1) / G, H};
        const int B = 3, Bv = B * qs.NG;
        std::vector<int> seen((size_t)B * T * H, 0);
        for (int r = 0; r < Bv; ++r) {
          const int tl = qs.last_token(r);
          CHECK(tl >= 0 && tl < T && tl >= (r % qs.NG) * G, "H=%d T=%d r=%d tl=%d", H, T, r, tl);
          for (int v = 0; v < 128; ++v) {
            const int t = qs.token(r, v), h = v % H, b = r / qs.NG;
            if (t >= T) {
              CHECK(qs.shift(r, v) >= (1 << 30), "H=%d T=%d r=%d v=%d: padding lane", H, T, r, v);
              continue;
            }
            ++seen[((size_t)b * T + t) * H + h];
            CHECK(qs.qrow(r) + v == ((long long)b * T + t) * H + h, "H=%d T=%d r=%d v=%d", H, T, r, v);
            // query t sits at position n - T + t; the virtual row's view ends at n - T + tl
            CHECK(qs.shift(r, v) == tl - t && t <= tl, "H=%d T=%d r=%d v=%d", H, T, r, v);
          }
        }
        bool once = true;
        for (int c : seen) once = once && c == 1;
        CHECK(once, "H=%d T=%d: a (row, token, head) not covered exactly once", H, T);
      }
  }
  std::printf("%d\n", fails);
  return fails != 0;
}
"""


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_scheduling_host_logic(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    src = tmp_path / "host_logic.cu"
    src.write_text(HARNESS)
    exe = tmp_path / "host_logic"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "--expt-relaxed-constexpr",
                        "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("0"), run.stdout[-2000:]
