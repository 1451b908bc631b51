"""The varlen plan's bounds on a malformed cu_seqlens, checked on the CPU.

cu_seqlens is device-resident and unchecked before the launch.  The kernels that read it take
every sequence's range and every chunk-table index through the helpers of csrc/kda_plan.h,
which clamp them into [0, T] and into the table.  A host restatement of the plan kernel (the
same helpers, the same loop bounds) runs here on malformed arrays, and the test checks that no
table write or token access leaves its buffer, that exactly the malformed arrays are flagged,
and that a valid array gives the plain chunk table.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

from gated_delta_rule_23_gb300 import _native

DRIVER = r"""
#include <cstdio>
#include <vector>
#include "kda_plan.h"
using namespace kda;
// Reads cases "N T v0 .. vN" from stdin; for each prints
//   bad used max_write_index min_token max_token_end rec_max_slot_end
int main() {
    int N; long long T;
    while (std::scanf("%d %lld", &N, &T) == 2) {
        std::vector<int64_t> cu(N + 1);
        for (auto &x : cu) { long long v; std::scanf("%lld", &v); x = v; }
        const int64_t cap = varlen_chunk_capacity(N, T);
        // the plan kernel: counts, exclusive scan, bounded table writes
        bool bad = false;
        std::vector<int64_t> off(N + 1);
        int64_t carry = 0;
        for (int n = 0; n < N; ++n) {
            int64_t b, l;
            bad |= seq_range(cu.data(), n, N, T, b, l);
            off[n] = carry;
            carry += seq_chunks(l);
        }
        off[N] = carry;
        const int64_t used = carry < cap ? carry : cap;
        bad |= carry > cap;
        int64_t max_w = -1, min_tok = T, max_end = 0;
        for (int64_t c = 0; c < used; ++c) {
            const int s = owner_of_chunk(off.data(), N, c);
            int64_t b, l;
            seq_range(cu.data(), s, N, T, b, l);
            const int64_t tok0 = b + (c - off[s]) * PLAN_CHUNK, rem = b + l - tok0;
            const int64_t end = tok0 + (rem < PLAN_CHUNK ? rem : PLAN_CHUNK);   // the prep CTA's tokens
            if (c > max_w) max_w = c;
            if (rem > 0) { if (tok0 < min_tok) min_tok = tok0; if (end > max_end) max_end = end; }
        }
        for (int64_t c = used; c < cap; ++c)
            if (c > max_w) max_w = c;
        // the recurrence kernel: per sequence, chunks clamped to the table
        int64_t rec_end = 0;
        for (int n = 0; n < N; ++n) {
            int64_t b, l;
            seq_range(cu.data(), n, N, T, b, l);
            const int64_t usable = usable_chunks(off[n], seq_chunks(l), cap);
            if (usable * PLAN_CHUNK < l) l = usable * PLAN_CHUNK;
            const int64_t e = off[n] + seq_chunks(l);
            if (l > 0) {
                if (e > rec_end) rec_end = e;
                if (b < min_tok) min_tok = b;
                if (b + l > max_end) max_end = b + l;
            }
        }
        std::printf("%d %lld %lld %lld %lld %lld\n", (int)bad, (long long)used, (long long)max_w,
                    (long long)min_tok, (long long)max_end, (long long)rec_end);
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def driver():
    d = tempfile.mkdtemp(prefix="kda_plan_")
    src, exe = os.path.join(d, "plan.cpp"), os.path.join(d, "plan")
    open(src, "w").write(DRIVER)
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", _native.CSRC, "-o", exe, src], check=True)
    return exe


def run(driver, cases):
    text = "".join(f"{len(cu) - 1} {T} " + " ".join(str(int(x)) for x in cu) + "\n" for cu, T in cases)
    out = subprocess.run([driver], input=text, capture_output=True, text=True, check=True).stdout.split("\n")
    return [tuple(int(x) for x in ln.split()) for ln in out if ln.strip()]


def valid(cu, T):
    cu = np.asarray(cu)
    return cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)


def test_malformed_cu_seqlens_stay_in_bounds(driver):
    rng = np.random.default_rng(7)
    cases = [([0, 100, 50, 150], 150), ([0, 8192, 0, 8192], 8192), ([-5, 10, 20], 20), ([0, 10, 30], 20),
             ([5, 10, 20], 20), ([0, 1 << 40, 3], 3), ([0, -1 << 40, 7], 7), ([0, 0], 0), ([0, 64, 128], 128)]
    for _ in range(300):
        N = int(rng.integers(1, 12))
        T = int(rng.integers(0, 3000))
        cu = np.sort(rng.integers(0, T + 1, N + 1))
        cu[0], cu[-1] = 0, T
        kind = rng.integers(0, 4)
        if kind == 1:
            cu = rng.integers(-200, T + 200, N + 1)
        elif kind == 2:
            cu[rng.integers(0, N + 1)] += int(rng.integers(-500, 500))
        cases.append((cu, T))
    for (cu, T), (bad, used, max_w, min_tok, max_end, rec_end) in zip(cases, run(driver, cases)):
        N = len(cu) - 1
        cap = (T + 63 * N) // 64
        assert bad == (not valid(cu, T)), (cu, T)
        assert max_w < cap and used <= cap            # chunk-table writes stay in the table
        assert rec_end <= cap                         # the recurrence's slots stay in the workspace
        assert 0 <= min_tok and max_end <= T          # tokens read and written stay in [0, T)


def test_valid_cu_seqlens_give_the_plain_table(driver):
    cu = [0, 1, 65, 65, 300, 1000]
    (bad, used, max_w, min_tok, max_end, rec_end), = run(driver, [(cu, 1000)])
    chunks = sum(-(-(b - a) // 64) for a, b in zip(cu[:-1], cu[1:]))
    assert bad == 0 and used == chunks == rec_end and min_tok == 0 and max_end == 1000


def _bitonic_order(lengths):
    """The plan kernel's longest-first order restated: keys length * 4096 + (4095 - index), padded with -1 to
    m = the power of two from N up (at least 2), sorted descending by the same compare-exchange network
    (stage (k, j): thread t < m / 2 pairs i = 2 j (t / j) + t % j with i + j, descending where i & k == 0)."""
    N = len(lengths)
    m = 2
    while m < N:
        m <<= 1
    keys = [int(lengths[s]) * 4096 + (4095 - s) if s < N else -1 for s in range(m)]
    k = 2
    while k <= m:
        j = k >> 1
        while j > 0:
            for t in range(m >> 1):
                i = 2 * j * (t // j) + t % j
                x, y = keys[i], keys[i + j]
                if (x < y) if (i & k) == 0 else (x > y):
                    keys[i], keys[i + j] = y, x
            j >>= 1
        k <<= 1
    return [4095 - (key & 4095) for key in keys[:N]]


@pytest.mark.parametrize("N", [2, 3, 5, 12, 16, 17, 100, 257])
def test_longest_first_order_network(N):
    """The sort network sized to the sequence count orders the sequences longest first, ties by index."""
    rng = np.random.default_rng(N)
    lengths = rng.integers(0, 50, size=N)   # many ties
    want = sorted(range(N), key=lambda s: (-int(lengths[s]), s))
    assert _bitonic_order(lengths) == want
