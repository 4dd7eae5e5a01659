"""A sharded optimizer step from Python: the example the README shows, as a file that runs.

The same calls exist in C (include/zs.h).  run() returns the buffers so a test can check them.
"""

import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs


def run():
    shapes = [(4096, 1024), (1024,), (1024, 4096)]                 # the model's parameters, in order
    plan = zs.Plan(shapes, n_d=8, stage=zs.ZS_STAGE_ZERO2, bucket_bytes=25 << 20)
    P = plan.padded                                               # flat length, a multiple of N_d
    grads = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(8)]      # per rank
    replicas = [torch.zeros(P, dtype=torch.bfloat16, device="cuda") for _ in range(8)]   # per rank
    master = torch.zeros(P, device="cuda")                        # fp32 shards of all ranks, rank-major
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    hp = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}
    # ... fill grads[q] with rank q's gradients, master with the initial weights ...
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, replicas, hp, step=1)
    # or bucket by bucket as gradients become ready, last bucket first:
    zs.zs_fused_step_buckets(plan, [plan.n_buckets - 1], grads, master, m, v, replicas, hp, step=2)
    return {"plan": plan, "grads": grads, "replicas": replicas, "master": master, "m": m, "v": v}


if __name__ == "__main__":
    out = run()
    torch.cuda.synchronize()
    print("stepped %d parameters on %d simulated ranks" % (out["plan"].numel, out["plan"].n_d))
