"""The SnapKV scoring kernel's work cut, modelled on the host.

The prefill scoring launch (csrc/prefill_score.cu) lays its (sequence, KV head, resident
block) triples end to end, each (sequence, KV head) group led by a fixed charge for the
costs of a run, and gives CTA c the share [c T / G, (c + 1) T / G) of that weighted
order.  Each share is cut into runs, and phase 2 cuts runs into pieces of at most 62
blocks plus a halo block on each side (the pool's reach of 3 positions stays within one
neighbouring block).  This model restates those rules and checks the properties the
kernel relies on: every block is scored once per phase, each piece streams its halo,
every CTA below G holds a block, a CTA's row partials land in a slot (CTA + group) that no
other (CTA, group) pair uses, and the closed form for a group's first and last CTA, which
the statistics warp waits on, names exactly the CTAs that publish for the group.
"""
import os
import random
import re

import pytest

BLOCKS_PER_STAGE = 8
PIECE_MAX = 62
RUN_COST = 12                      # the kernel's charge per group, in blocks


def layout(n_blocks, charge):
    """Weighted start of each sequence: a sequence with n > 0 blocks weighs n + charge."""
    off = [0]
    for n in n_blocks:
        off.append(off[-1] + (n + charge if n > 0 else 0))
    return off


def stages(off, hkv, charge, x0, x1):
    """The stages one CTA streams for the share [x0, x1), in order."""
    n_seqs = len(off) - 1
    st = {}

    def start_run(x):
        lo, hi = 0, n_seqs - 1
        while lo < hi:                                  # last slot starting at or before x
            mid = (lo + hi + 1) // 2
            if hkv * off[mid] <= x:
                lo = mid
            else:
                hi = mid - 1
        w = off[lo + 1] - off[lo]
        n = w - charge
        base = hkv * off[lo]
        kvh = (x - base) // w
        gs = base + kvh * w + charge                    # the group's first block
        i1 = min(x1 - gs, n)
        p0 = max(x - gs, 0)
        if i1 <= p0:
            return False
        st.update(sl=lo, kvh=kvh, n=n, gs=gs, i1=i1, p0=p0, first=True)
        start_piece()
        return True

    def start_piece():
        if st["phase"] == 0:
            st.update(p1=st["i1"], v0=st["p0"], e=st["i1"])
        else:
            st["p1"] = min(st["p0"] + PIECE_MAX, st["i1"])
            st["v0"] = max(st["p0"] - 1, 0)
            st["e"] = min(st["p1"] + 1, st["n"])
        st["b"] = st["v0"]

    st["phase"] = 0
    out = []
    live = x0 < x1 and start_run(x0)
    while live:
        nb = min(BLOCKS_PER_STAGE, st["e"] - st["b"])
        s = dict(phase=st["phase"], g=st["sl"] * hkv + st["kvh"], n=st["n"], gs=st["gs"], b0=st["b"], nb=nb,
                 c0=st["p0"], c1=st["p1"], run_first=st["first"], run_last=False)
        st["first"] = False
        st["b"] += nb
        s["piece_last"] = st["b"] >= st["e"]
        if s["piece_last"]:
            if st["phase"] == 1 and st["p1"] < st["i1"]:
                st["p0"] = st["p1"]
                start_piece()
            else:
                s["run_last"] = True
                x = st["gs"] + st["i1"]
                if x < x1 and start_run(x):
                    pass
                elif st["phase"] == 0:
                    st["phase"] = 1
                    start_run(x0)
                else:
                    live = False
        out.append(s)
    return out


def check_cut(n_blocks, hkv, grid, charge):
    off = layout(n_blocks, charge)
    T = hkv * off[-1]
    if T == 0:
        return
    G = min(grid, max(1, T // (charge + 4)))
    scored = [dict(), dict()]
    publishers, slots = {}, set()
    for c in range(G):
        x0, x1 = c * T // G, (c + 1) * T // G
        S = stages(off, hkv, charge, x0, x1)
        assert S, "CTA %d of %d holds no block" % (c, G)
        assert [s["phase"] for s in S] == sorted(s["phase"] for s in S)
        for s in S:
            assert 1 <= s["nb"] <= BLOCKS_PER_STAGE
            if s["phase"] == 0:
                for b in range(s["b0"], s["b0"] + s["nb"]):
                    scored[0][(s["g"], b)] = scored[0].get((s["g"], b), 0) + 1
                if s["run_last"]:
                    assert c + s["g"] not in slots
                    slots.add(c + s["g"])
                    publishers.setdefault(s["g"], set()).add(c)
            elif s["piece_last"]:
                assert s["c1"] - s["c0"] <= PIECE_MAX
                for b in range(s["c0"], s["c1"]):
                    scored[1][(s["g"], b)] = scored[1].get((s["g"], b), 0) + 1
        # phase 2 streams each piece with one halo block on each side, where there is one
        for s in S:
            if s["phase"] == 1 and s["piece_last"]:
                assert s["b0"] + s["nb"] == min(s["c1"] + 1, s["n"])
    for sl, n in enumerate(n_blocks):
        for kvh in range(hkv):
            g = sl * hkv + kvh
            for b in range(n):
                assert scored[0].get((g, b)) == 1 and scored[1].get((g, b)) == 1, (g, b)
            if n:
                gs = hkv * off[sl] + kvh * (n + charge) + charge
                first, last = ((gs + 1) * G - 1) // T, ((gs + n) * G - 1) // T
                assert publishers[g] == set(range(first, last + 1))


def test_cut_of_the_32k_context_batch():
    """16 sequences x 4 KV heads x 257 resident blocks (4096 entries plus the next block)."""
    for charge in (0, RUN_COST):
        check_cut([257] * 16, 4, 152, charge)


@pytest.mark.parametrize("charge", [0, 3, RUN_COST, 20])
def test_cut_of_ragged_batches(charge):
    rng = random.Random(charge)
    for _ in range(150):
        n_blocks = [rng.choice([0, 1, 2, 5, 16, 63, 64, 65, 200, 257, 600]) for _ in range(rng.randint(1, 40))]
        check_cut(n_blocks, rng.choice([1, 4, 8]), rng.choice([1, 2, 7, 152]), charge)


def test_cut_of_single_block_sequences():
    check_cut([1] * 512, 8, 152, RUN_COST)
    check_cut([0, 0, 1, 0], 1, 152, RUN_COST)


def test_model_uses_the_kernels_charge():
    src = os.path.join(os.path.dirname(__file__), "..", "attention_scored_kv_gb300", "csrc", "prefill_score.cu")
    m = re.search(r"constexpr int kRunCost = (\d+);", open(src).read())
    assert m and int(m.group(1)) == RUN_COST
