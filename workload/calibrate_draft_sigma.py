"""Choose the draft noise of the MTP verify batch so that the drafts' top-k
sets overlap token 0's by about one half, as the workload asks.

Routes token 0 and its three drafts through the first layer's router with
the oracle, for a grid of sigma, over many seeded input sets, and prints the
mean |S_0 & S_i| / k.  Usage: python -m workload.calibrate_draft_sigma
"""
import sys

import numpy as np

import oracle
import workload as W


def mean_overlap(cfg, sigma, n_sets=64, layer=0):
    Wr, b = W.router(cfg, layer)
    c = cfg.replace(draft_sigma=sigma)
    tot = []
    for i in range(n_sets):
        x = W.activations(c, index=i)
        z = oracle.router_logits(Wr, b, x)
        ids, _, _ = oracle.topk_softmax(z, cfg.top_k)
        s0 = set(ids[0])
        tot += [len(s0 & set(ids[t])) / cfg.top_k for t in range(1, x.shape[0])]
    return float(np.mean(tot))


def main():
    cfg = W.CONFIGS["mtp35b"]
    for sigma in [float(s) for s in sys.argv[1:]] or [0.1, 0.5, 1.0, 1.4, 1.6, 1.8, 2.0]:
        print("sigma %.3f  mean overlap %.3f" % (sigma, mean_overlap(cfg, sigma)))


if __name__ == "__main__":
    main()
