"""Seeded synthetic inputs and the parameter lists of the benchmarked model shapes.

This module holds none of the method's arithmetic: it only names parameter
shapes and draws random tensors.  Both the CUDA path (bench, tests) and the
oracle side of the tests take their inputs from here.  It stands apart from
the library package and imports nothing but torch, so a process that feeds
the oracle from it (the CPU baseline, the oracle tests) never loads the
library it checks.

Shapes (random-initialised stand-ins; no weights or datasets are used):

* ``mlp-tiny``   2-layer MLP: W1 256x512, b1 512, W2 512x256, b2 256 (262,912).
* ``gpt2-small`` 12 layers, d=768, ffn 3072, vocab 50257, learned positions
                 n_ctx=1024, tied embeddings, LayerNorms with bias
                 (124,439,808).
* ``llama-1.3b`` 24 layers, d=2048, SwiGLU ffn 5504, 16 heads (MHA), RMSNorm,
                 vocab 32000, untied output (1,345,423,360).  ``llama-1.3b-units``
                 is the same list grouped one unit per layer plus a root unit
                 (embedding, final norm, output), for ZeRO-3 and FSDP2 groups.
* ``llama-small-units`` 4 layers, d=1024, ffn 2816, vocab 32000, untied, one
                 unit per layer plus the root unit (116,925,440): the same kernels as
                 the Llama-1.3B grouping on a few GB, for profiler captures.
* ``llama-7b``   32 layers, d=4096, ffn 11008, vocab 32000, untied
                 (6,738,415,616); one FSDP unit per layer plus a root unit
                 holding the embedding, final norm and output.
* ``flat-2^28+7`` one flat tensor of 2^28 + 7 elements (padding sweep).

Draws: gradients are bf16 values of N(0, sigma) in fp32, optionally with an
independent Bernoulli(p) mask multiplying entries by a factor before the
cast; master weights are N(0, 0.02) fp32; padding elements are zero in every
buffer.  Generators are keyed by (seed, step, rank).
"""

import torch


def _layer_gpt2(d=768, ffn=3072):
    return [(d,), (d,), (d, 3 * d), (3 * d,), (d, d), (d,), (d,), (d,), (d, ffn), (ffn,), (ffn, d), (d,)]


def _layer_llama(d, ffn):
    return [(d,), (d, d), (d, d), (d, d), (d, d), (d,), (ffn, d), (ffn, d), (d, ffn)]


def workload_params(name):
    """(shapes, unit_of_param or None) of a named model shape, in module order."""
    if name == "mlp-tiny":
        return [(256, 512), (512,), (512, 256), (256,)], None
    if name == "gpt2-small":
        shapes = [(50257, 768), (1024, 768)]
        for _ in range(12):
            shapes += _layer_gpt2()
        shapes += [(768,), (768,)]
        return shapes, None
    if name in ("llama-1.3b", "llama-1.3b-units"):
        n_layers = 24
        shapes, units = [(32000, 2048)], [n_layers]
        for layer in range(n_layers):
            ls = _layer_llama(2048, 5504)
            shapes += ls
            units += [layer] * len(ls)
        shapes += [(2048,), (32000, 2048)]
        units += [n_layers, n_layers]
        return shapes, (units if name == "llama-1.3b-units" else None)
    if name == "llama-small-units":
        n_layers = 4
        shapes, units = [(32000, 1024)], [n_layers]
        for layer in range(n_layers):
            ls = _layer_llama(1024, 2816)
            shapes += ls
            units += [layer] * len(ls)
        shapes += [(1024,), (32000, 1024)]
        units += [n_layers, n_layers]
        return shapes, units
    if name == "llama-7b":
        n_layers = 32
        shapes, units = [(32000, 4096)], [n_layers]
        for layer in range(n_layers):
            ls = _layer_llama(4096, 11008)
            shapes += ls
            units += [layer] * len(ls)
        shapes += [(4096,), (32000, 4096)]
        units += [n_layers, n_layers]
        return shapes, units
    if name == "flat-2^28+7":
        return [(2 ** 28 + 7,)], None
    raise KeyError(name)


def _gen(device, seed, step, rank):
    g = torch.Generator(device=device)
    g.manual_seed(((int(seed) * 1_000_003 + int(step)) * 10_007 + int(rank)) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _row_stride(padded):
    return (int(padded) + 63) // 64 * 64


def rank_buffers(n_d, padded, dtype, device):
    """N_d zeroed rank buffers of `padded` elements, each 16-byte aligned (rows of one allocation)."""
    stride = _row_stride(padded)
    base = torch.zeros((n_d, stride), dtype=dtype, device=device)
    return [base[q, :padded] for q in range(n_d)], base


def fill_grads(bufs, pad_ranges, seed, step, sigma, outlier_p=0.0, outlier_scale=100.0, chunk=1 << 27):
    """Fill each rank's bf16 buffer with N(0, sigma) (times outlier_scale on a Bernoulli(outlier_p) mask)."""
    for q, buf in enumerate(bufs):
        g = _gen(buf.device, seed, step, q)
        n = buf.numel()
        for lo in range(0, n, chunk):
            hi = min(n, lo + chunk)
            x = torch.randn(hi - lo, generator=g, device=buf.device, dtype=torch.float32) * sigma
            if outlier_p > 0:
                mask = torch.rand(hi - lo, generator=g, device=buf.device) < outlier_p
                x = torch.where(mask, x * outlier_scale, x)
            buf[lo:hi].copy_(x.to(torch.bfloat16))
        for lo, hi in pad_ranges:
            buf[lo:hi].zero_()
    return bufs


def rank_grads(n_d, padded, pad_ranges, seed, step, sigma, outlier_p=0.0, device="cpu"):
    bufs, base = rank_buffers(n_d, padded, torch.bfloat16, device)
    fill_grads(bufs, pad_ranges, seed, step, sigma, outlier_p)
    return bufs, base


def master_init(padded, pad_ranges, seed, device="cpu", sigma=0.02, chunk=1 << 27):
    out = torch.empty(_row_stride(padded), dtype=torch.float32, device=device)[:padded]
    g = _gen(out.device, seed, 0, 1_000_000)
    for lo in range(0, padded, chunk):
        hi = min(padded, lo + chunk)
        out[lo:hi].copy_(torch.randn(hi - lo, generator=g, device=out.device) * sigma)
    for lo, hi in pad_ranges:
        out[lo:hi].zero_()
    return out


def zeros_f32(padded, device="cpu"):
    return torch.zeros(_row_stride(padded), dtype=torch.float32, device=device)[:padded]


# Per-configuration settings of the benchmarked workloads.
WORKLOADS = {
    "mlp-tiny-zero1": dict(model="mlp-tiny", n_d=4, stage=1, bucket_bytes=0, sigma=1e-3, outlier_p=0.0,
                           seed=0, steps=10, micro=1),
    "gpt2-small-zero1": dict(model="gpt2-small", n_d=8, stage=1, bucket_bytes=25 << 20, sigma=1e-3,
                             outlier_p=0.0, seed=1, steps=1, micro=4),
    "llama-1.3b-zero2": dict(model="llama-1.3b", n_d=8, stage=2, bucket_bytes=25 << 20, sigma=5e-4,
                             outlier_p=1e-3, seed=2, steps=1, micro=1),
    "llama-7b-zero3": dict(model="llama-7b", n_d=16, stage=3, bucket_bytes=0, sigma=5e-4, outlier_p=0.0,
                           seed=3, steps=1, micro=1),
    "flat-sweep": dict(model="flat-2^28+7", n_d=8, stage=2, bucket_bytes=1 << 20, sigma=1e-3, outlier_p=0.0,
                       seed=4, steps=1, micro=1, sweep_n_d=(2, 4, 8, 16, 32),
                       sweep_bucket_mib=(1, 4, 16, 64, 256, 1024)),
}

HPARAMS = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}
