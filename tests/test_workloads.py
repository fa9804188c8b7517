"""The synthetic workloads have the structure their descriptions give: the skewed-load
configuration's busiest expert takes about 10x the mean load (routing by the oracle on
that workload's own inputs), and the seeded generators are reproducible."""

import numpy as np

import oracle
import workloads


def test_skewed_workload_hot_expert_load_is_about_10x_mean():
    cfg = workloads.SKEWED
    x = workloads.gen_x(cfg).float().numpy()
    z = oracle.router_logits(x, workloads.gen_centroids(cfg).numpy())
    idx, _ = oracle.route(z, workloads.gen_bias(cfg).numpy(), cfg.n_groups, cfg.topk_groups,
                          cfg.group_topn, cfg.K)
    cnt = np.bincount(idx.ravel(), minlength=cfg.E)
    assert cnt.sum() == cfg.T * cfg.K
    assert 9.5 <= cnt.max() / cnt.mean() <= 10.5
    assert (cnt > 0).sum() < cfg.E                   # some experts idle, as popularity is skewed


def test_generators_are_reproducible():
    cfg = workloads.TINY
    assert np.array_equal(workloads.gen_x(cfg).float().numpy(),
                          workloads.gen_x(cfg).float().numpy())
    assert np.array_equal(workloads.gen_bias(cfg).numpy(), workloads.gen_bias(cfg).numpy())
