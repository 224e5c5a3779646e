"""Seeded synthetic inputs for the five error-feedback workloads.

This module produces inputs only: parameter-set shapes, per-tensor k from a
keep ratio, and seeded random gradients / weights.  It holds none of the
error-feedback arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.

The pages measure on ResNet-50 / ImageNet and BERT training runs
("梯度稀疏化：只传输重要的梯度元素" §实验效果与适用边界; "1bit Adam梯度压缩技术原理与
分布式训练优化" §5.1).  Those need datasets and trained models, so synthetic
tensors with the same shapes and heavy-tailed value distributions stand in
for real gradients.

Workloads (sizes, distributions, k and step counts):

* ``topk_2p20``   one fp32 tensor, n = 2**20, Student-t(3) x 1e-3, k = 1 %
                   (10 486), 3 steps, W = 1, SGD eta = 0.1 on w0 ~ N(0, 0.02).
* ``sign_2p24``   one fp32 tensor, n = 2**24, N(0, 1e-3) (std), beta1 = 0.9,
                   10 steps of 1-bit EF followed by the 1-bit momentum.
* ``resnet50``    161 ResNet-50 parameter tensors (25 557 032 elements);
                   each tensor has one scale s_t = exp(-7 + Z_t) fixed across
                   steps and fresh N(0, 1) per step; k = 0.1 % of tensors with
                   at least 1 000 000 elements, else 1 %, at least 1; 3 steps.
* ``bert_large``  BERT-large parameters flattened into one vector
                   (335 141 888 elements), W = 8 workers each drawing
                   Laplace(0, b = 1e-4) per step, top-0.1 % (335 142), the
                   packets summed into a dense gradient, SGD eta = 1e-3,
                   w0 ~ N(0, 0.02), 3 steps.
* ``slab_2p31``   one flat slab, n = 2**31, Student-t(3) x 1e-3, W = 4,
                   top-0.1 % (2 147 484) with int32 indices and with a bitmap,
                   plus 1-bit EF (beta1 = 0.9) on the same gradients, each
                   aggregated locally with SGD eta = 0.1; 2 steps.

Seeds: ``seed(config, worker, step) = 1_000_000 * config + 1_000 * worker +
step`` with configs numbered 1-5 in the order above.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence, Tuple

import torch

# ---------------------------------------------------------------------------
# parameter-set shapes
# ---------------------------------------------------------------------------


def resnet50_param_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    """The 161 trainable tensors of ResNet-50 in definition order.

    Stem conv 64x3x7x7 + BN; four bottleneck stages (width, blocks, out) =
    (64, 3, 256), (128, 4, 512), (256, 6, 1024), (512, 3, 2048), each block
    conv1 width x in x 1 x 1, conv2 width x width x 3 x 3, conv3
    out x width x 1 x 1, a BN (weight, bias) after every conv, and in block 0
    a downsample conv out x in x 1 x 1 + BN; then fc 1000 x 2048 + bias.
    """
    shapes: List[Tuple[str, Tuple[int, ...]]] = []

    def bn(prefix: str, c: int) -> None:
        shapes.append((prefix + ".weight", (c,)))
        shapes.append((prefix + ".bias", (c,)))

    shapes.append(("conv1.weight", (64, 3, 7, 7)))
    bn("bn1", 64)
    cin = 64
    for si, (width, blocks, out) in enumerate(
            [(64, 3, 256), (128, 4, 512), (256, 6, 1024), (512, 3, 2048)], 1):
        for b in range(blocks):
            p = f"layer{si}.{b}"
            shapes.append((p + ".conv1.weight", (width, cin, 1, 1)))
            bn(p + ".bn1", width)
            shapes.append((p + ".conv2.weight", (width, width, 3, 3)))
            bn(p + ".bn2", width)
            shapes.append((p + ".conv3.weight", (out, width, 1, 1)))
            bn(p + ".bn3", out)
            if b == 0:
                shapes.append((p + ".downsample.0.weight", (out, cin, 1, 1)))
                bn(p + ".downsample.1", out)
            cin = out
    shapes.append(("fc.weight", (1000, 2048)))
    shapes.append(("fc.bias", (1000,)))
    return shapes


def bert_large_param_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    """BERT-large (24 layers, hidden 1024, FFN 4096, vocab 30522, 512
    positions, 2 token types) parameters including biases, LayerNorms and the
    pooler: 335 141 888 elements."""
    h, f, L = 1024, 4096, 24
    shapes: List[Tuple[str, Tuple[int, ...]]] = [
        ("embeddings.word", (30522, h)),
        ("embeddings.position", (512, h)),
        ("embeddings.token_type", (2, h)),
        ("embeddings.ln.weight", (h,)),
        ("embeddings.ln.bias", (h,)),
    ]
    for i in range(L):
        p = f"layer{i}"
        for name in ("query", "key", "value", "attn_out"):
            shapes.append((f"{p}.{name}.weight", (h, h)))
            shapes.append((f"{p}.{name}.bias", (h,)))
        shapes.append((f"{p}.attn_ln.weight", (h,)))
        shapes.append((f"{p}.attn_ln.bias", (h,)))
        shapes.append((f"{p}.intermediate.weight", (f, h)))
        shapes.append((f"{p}.intermediate.bias", (f,)))
        shapes.append((f"{p}.output.weight", (h, f)))
        shapes.append((f"{p}.output.bias", (h,)))
        shapes.append((f"{p}.out_ln.weight", (h,)))
        shapes.append((f"{p}.out_ln.bias", (h,)))
    shapes.append(("pooler.weight", (h, h)))
    shapes.append(("pooler.bias", (h,)))
    return shapes


def numel(shape: Sequence[int]) -> int:
    return int(math.prod(shape))


def k_from_ratio(n: int, num: int, den: int) -> int:
    """k for keep ratio num/den of n elements, rounded half up, at least 1.

    Integer arithmetic: max(1, (n * num + den // 2) // den).  For n = 0 the
    result is 0 (an empty tensor selects nothing).
    """
    if n <= 0:
        return 0
    return max(1, (n * num + den // 2) // den)


def segments_from_sizes(sizes: Sequence[int]) -> List[int]:
    """Flat-buffer offsets (nseg + 1 entries) for consecutive tensors."""
    offs = [0]
    for s in sizes:
        offs.append(offs[-1] + int(s))
    return offs


def resnet50_segments() -> Tuple[List[int], List[int]]:
    """(offsets, k) of the layerwise ResNet-50 workload: 0.1 % for tensors of
    at least 1 000 000 elements, else 1 %, minimum 1."""
    sizes = [numel(s) for _, s in resnet50_param_shapes()]
    ks = [k_from_ratio(n, 1, 1000) if n >= 1_000_000 else k_from_ratio(n, 1, 100)
          for n in sizes]
    return segments_from_sizes(sizes), ks


# ---------------------------------------------------------------------------
# seeded generators
# ---------------------------------------------------------------------------

_CHUNK = 1 << 26  # elements per generator call for very large tensors


def seed(config: int, worker: int = 0, step: int = 0) -> int:
    return 1_000_000 * config + 1_000 * worker + step


def _gen(seed_: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed_))
    return g


def normal(n: int, std: float, seed_: int, device="cpu",
           out: torch.Tensor | None = None) -> torch.Tensor:
    """n fp32 draws of N(0, std**2)."""
    gen = _gen(seed_, device)
    out = torch.empty(n, dtype=torch.float32, device=device) if out is None else out
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        torch.randn(b - a, generator=gen, device=device, dtype=torch.float32,
                    out=out[a:b])
        out[a:b].mul_(std)
    return out


def student_t3(n: int, scale: float, seed_: int, device="cpu",
               out: torch.Tensor | None = None) -> torch.Tensor:
    """n fp32 draws of scale * T with T ~ Student-t(3 d.o.f.):
    T = Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3), all Z standard normal."""
    gen = _gen(seed_, device)
    out = torch.empty(n, dtype=torch.float32, device=device) if out is None else out
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        m = b - a
        z = torch.randn(4, m, generator=gen, device=device, dtype=torch.float32)
        chi2 = z[1].square() + z[2].square() + z[3].square()
        out[a:b] = z[0] / torch.sqrt(chi2 / 3.0) * scale
        del z, chi2
    return out


def laplace(n: int, b: float, seed_: int, device="cpu",
            out: torch.Tensor | None = None) -> torch.Tensor:
    """n fp32 draws of Laplace(0, b) as b * (E1 - E2), E ~ Exp(1)."""
    gen = _gen(seed_, device)
    out = torch.empty(n, dtype=torch.float32, device=device) if out is None else out
    for a in range(0, n, _CHUNK):
        m = min(n, a + _CHUNK) - a
        e = torch.empty(2, m, device=device, dtype=torch.float32)
        e.exponential_(1.0, generator=gen)
        out[a:a + m] = (e[0] - e[1]) * b
        del e
    return out


def lognormal_scaled_normal(sizes: Sequence[int], scale_seed: int, seed_: int,
                            device="cpu") -> torch.Tensor:
    """Concatenated per-tensor gradients s_t * N(0, 1) with one scale per
    tensor, s_t = exp(-7 + Z_t): the scales come from ``scale_seed`` (fixed
    across steps), the N(0, 1) draws from ``seed_`` (fresh per step)."""
    zs = torch.randn(len(sizes), generator=_gen(scale_seed, "cpu"),
                     dtype=torch.float64)
    scales = torch.exp(-7.0 + zs).tolist()
    total = int(sum(sizes))
    out = normal(total, 1.0, seed_, device)
    a = 0
    for s, n in zip(scales, sizes):
        out[a:a + n].mul_(float(s))
        a += n
    return out


# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    config: int              # 1..5, also the seed family
    n: int                   # elements per worker
    workers: int
    steps: int
    seg_offsets: Tuple[int, ...]
    seg_k: Tuple[int, ...]
    grad: str                # "student_t3" | "normal" | "laplace" | "lognormal"
    grad_scale: float
    eta: float = 0.0
    beta1: float = 0.9
    w0_std: float = 0.02

    @property
    def total_k(self) -> int:
        return int(sum(self.seg_k))

    def gradient(self, worker: int, step: int, device="cpu",
                 out: torch.Tensor | None = None) -> torch.Tensor:
        s = seed(self.config, worker, step)
        if self.grad == "student_t3":
            return student_t3(self.n, self.grad_scale, s, device, out)
        if self.grad == "normal":
            return normal(self.n, self.grad_scale, s, device, out)
        if self.grad == "laplace":
            return laplace(self.n, self.grad_scale, s, device, out)
        if self.grad == "lognormal":
            sizes = [self.seg_offsets[i + 1] - self.seg_offsets[i]
                     for i in range(len(self.seg_k))]
            g = lognormal_scaled_normal(sizes, seed(self.config, worker, 999), s,
                                        device)
            if out is not None:
                out.copy_(g)
                return out
            return g
        raise ValueError(self.grad)

    def weights(self, device="cpu") -> torch.Tensor:
        return normal(self.n, self.w0_std, seed(self.config, 999, 0), device)


def _single(n: int, num: int, den: int) -> Tuple[Tuple[int, ...], Tuple[int, ...]]:
    return (0, n), (k_from_ratio(n, num, den),)


def workload(name: str, n: int | None = None) -> Workload:
    """The named workload; ``n`` shrinks a single-segment workload (same
    distribution and ratio) for quick parity cases."""
    if name == "topk_2p20":
        n = 1 << 20 if n is None else n
        offs, ks = _single(n, 1, 100)
        return Workload(name, 1, n, 1, 3, offs, ks, "student_t3", 1e-3, eta=0.1)
    if name == "sign_2p24":
        n = 1 << 24 if n is None else n
        return Workload(name, 2, n, 1, 10, (0, n), (0,), "normal", 1e-3, beta1=0.9)
    if name == "resnet50":
        offs, ks = resnet50_segments()
        return Workload(name, 3, offs[-1], 1, 3, tuple(offs), tuple(ks),
                        "lognormal", 1.0, eta=0.1)
    if name == "bert_large":
        n = sum(numel(s) for _, s in bert_large_param_shapes()) if n is None else n
        offs, ks = _single(n, 1, 1000)
        return Workload(name, 4, n, 8, 3, offs, ks, "laplace", 1e-4, eta=1e-3)
    if name == "slab_2p31":
        n = 1 << 31 if n is None else n
        offs, ks = _single(n, 1, 1000)
        return Workload(name, 5, n, 4, 2, offs, ks, "student_t3", 1e-3, eta=0.1,
                        beta1=0.9)
    raise KeyError(name)


WORKLOADS = ("topk_2p20", "sign_2p24", "resnet50", "bert_large", "slab_2p31")
