"""The prefill GEMM's division of work, on the host (no GPU): the units that
q4_prefill_units lists come from the function the kernel itself runs.

The persistent prefill form (M > 128; C++ DeepSeek engine page §5.2, a
prompt's tokens as one matmul) runs 256 x 256 tiles round-robin; the tiles of
an incomplete last round pool their K steps into equal parts over the grid.
Checked here, for several shapes and SM counts:
  * every (tile, K step) is computed exactly once;
  * a CTA has at most one earlier part (role 2) and its last-step part
    (role 1) is its last unit, so the staging buffer it borrows is idle;
  * a last-step part adds exactly the parts that other CTAs hold of its tile,
    all of lower index;
  * run in CTA index order with only a few CTAs resident at a time, a
    last-step part never waits for a CTA that has not started, so every
    schedule finishes (the waits in the kernel are bounded, but must not be
    needed to end);
  * the parts of the tail are equal to within one K step.
"""

import pytest

import quantized_weight_q4_gb300 as q4

SHAPES = [(2048, 12288, 5120), (2304, 4352, 1024), (384, 2048, 5120), (2048, 12280, 1000),
          (1000, 3072, 2048), (300, 1000, 520), (513, 250, 1000), (2048, 5888, 520),
          (4096, 12288, 5120), (129, 256, 64), (256, 512, 64)]


def tiles_of(M, N):
    return -(-M // 256) * -(-N // 256)


def simulate(units, capacity):
    """Runs the CTAs in index order, `capacity` at a time: a role-2 unit
    completes at once, a role-1 unit once its helpers' role-2 units have;
    a CTA leaves when its units are done.  False if no CTA can move."""
    by_cta = {}
    for u in units:
        by_cta.setdefault(int(u[0]), []).append(u)
    ctas = sorted(by_cta)
    pos = {c: 0 for c in ctas}
    done2, resident, nxt, left = set(), [], 0, len(ctas)
    while left:
        while len(resident) < capacity and nxt < len(ctas):
            resident.append(ctas[nxt])
            nxt += 1
        moved = False
        for c in list(resident):
            us = by_cta[c]
            while pos[c] < len(us):
                role, c1, nc = int(us[pos[c]][6]), int(us[pos[c]][7]), int(us[pos[c]][8])
                if role == 1 and not all(h in done2 for h in range(c1, c1 + nc)):
                    break
                if role == 2:
                    done2.add(c)
                pos[c] += 1
                moved = True
            if pos[c] == len(us):
                resident.remove(c)
                left -= 1
                moved = True
        if not moved:
            return False
    return True


@pytest.mark.parametrize("sms", [152, 148, 20])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_prefill_units(M, N, K, sms):
    units = q4.q4_prefill_units(M, N, K, sms)
    ks = -(-K // 64)
    seen = set()
    tile_of = lambda u: (int(u[2]), int(u[3]))
    for u in units:
        for k in range(int(u[4]), int(u[5])):
            key = (tile_of(u), k)
            assert key not in seen, (M, N, K, sms, key)
            seen.add(key)
    assert len(seen) == tiles_of(M, N) * ks
    by_cta = {}
    for u in units:
        by_cta.setdefault(int(u[0]), []).append(u)
    assert len(by_cta) <= sms
    holders = {}   # tile -> CTAs holding an earlier part of it
    for c, us in by_cta.items():
        assert [int(u[1]) for u in us] == list(range(len(us)))
        assert sum(int(u[6]) == 2 for u in us) <= 1
        for i, u in enumerate(us):
            if int(u[6]) == 1:
                assert i == len(us) - 1, "a last-step part is its CTA's last unit"
                assert int(u[5]) == ks and int(u[4]) > 0
            if int(u[6]) == 2:
                assert int(u[5]) < ks
                holders.setdefault(tile_of(u), []).append(c)
            if int(u[6]) == 0:
                assert (int(u[4]), int(u[5])) == (0, ks)
    for c, us in by_cta.items():
        for u in us:
            if int(u[6]) == 1:
                helpers = list(range(int(u[7]), int(u[7]) + int(u[8])))
                assert sorted(holders.pop(tile_of(u))) == helpers
                assert all(h < c for h in helpers)
    assert not holders, "every earlier part has its last-step part"
    # equal parts of the tail
    tail = {}
    for u in units:
        if int(u[6]) != 0:
            tail[int(u[0])] = tail.get(int(u[0]), 0) + int(u[5]) - int(u[4])
    if tail:
        assert max(tail.values()) - min(tail.values()) <= 1
    for capacity in (1, 2, 5, sms):
        assert simulate(units, capacity), (M, N, K, sms, capacity)


def test_prefill_workload_shares_its_last_round():
    """M = 2048, K = 5120, N = 12288 on 152 SMs: 384 tiles, 304 of them whole
    (two rounds), the other 80 tiles' 6400 K steps in 152 parts."""
    units = q4.q4_prefill_units(2048, 12288, 5120, 152)
    whole = [u for u in units if int(u[6]) == 0]
    assert len(whole) == 304
    tail_ctas = {int(u[0]) for u in units if int(u[6]) != 0}
    assert len(tail_ctas) == 152
    assert sum(int(u[5]) - int(u[4]) for u in units if int(u[6]) != 0) == 80 * 80


def test_prefill_units_argument_errors():
    with pytest.raises(q4.Q4Error):
        q4.q4_prefill_units(128, 256, 64, 152)   # the prefill form starts above 128 rows
    with pytest.raises(q4.Q4Error):
        q4.q4_prefill_units(256, 256, 64, 0)
