"""CPU checks of the seeded workload generators the tests and the bench share:
the mixed-K large-verify layout (K_i in 1..15, whole requests under a row
limit, one draft flag and one random id per draft position) and the planted
cross-shard ties of the large-verify recipe."""
import numpy as np

import oracle
import workloads as wl


def test_mixed_k_layout_whole_requests():
    cu, flags, rand_ids = wl.draft_plan_mixed(6, 256, 15, 0.6, 202048)
    ks = np.diff(cu)
    assert cu[0] == 0 and ks.min() >= 1 and ks.max() <= 15
    assert len(np.unique(ks)) > 10                      # the lengths really vary
    assert flags.size == rand_ids.size == cu[-1]
    assert (rand_ids >= 0).all() and (rand_ids < 202048).all()
    c = wl.large_verify_mixed_k(rows_limit=300)
    n = c["cu_num_draft"].size - 1
    rows = c["logits"].shape[0]
    assert rows == int(c["cu_num_draft"][-1]) + n <= 300
    assert rows + int(ks[n]) + 1 > 300                  # the next request would not fit
    assert (c["cu_num_draft"] == cu[:n + 1]).all()
    assert c["flags"].size == c["rand_ids"].size == c["cu_num_draft"][-1]
    assert c["k"] == 15 and c["org_vocab"] == 202048


def test_mixed_k_planted_ties_resolve_to_the_lower_shard():
    c = wl.large_verify_mixed_k(rows_limit=250)
    x, shards = c["logits"], c["shards"]
    _, ids = oracle.full_argmax(x, c["org_vocab"])
    for r in range(0, x.shape[0], 100):
        s = 1 + (r // 100) % (len(shards) - 1)
        assert ids[r] == shards[s][0] - 1
