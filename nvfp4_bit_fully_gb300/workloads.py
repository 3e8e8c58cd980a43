"""Seeded synthetic inputs shaped like the pages' OLMo-2 70M-370M linear layers.

This module only draws random tensors (torch CPU generator, bf16 results); it
holds none of the method's arithmetic.  Tests, the bench and the oracle-side
checks all take their inputs from here so that both sides see identical bytes.

Workloads (named by what they are):
  tiny        X 256x512 N(0,1) with 8 fixed channels x50, W 512x512 N(0,0.02),
              dY 256x512 N(0,1e-3)
  quant_*     bf16 [R, C] N(0,1) with ceil(1%) of columns x30
  fwd_outctl  4 calibration batches X 16384x1024 N(0,1) with 20 fixed heavy
              channels x40, a fifth batch X, W 4096x1024 N(0,0.02)
  bwd_rht     dY 16384x4096 with heavy-tailed rows: row r = 1e-3 |T_r| N(0,1),
              T_r ~ Student-t(3); W 4096x1024 N(0,0.02); X 16384x1024 as quant_*
  layer_set   M=16384 tokens through QKV 1024->3072, out 1024->1024,
              gate/up 1024->8192, down 4096->1024; OsciReset master weights
"""
import math

import torch

LAYER_SET = (("qkv", 3072, 1024), ("out", 1024, 1024), ("gate_up", 8192, 1024), ("down", 1024, 4096))


def _gen(seed, stream=0):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000003 + int(stream))
    return g


def normal(shape, std, seed, stream=0):
    """bf16 N(0, std^2) tensor."""
    g = _gen(seed, stream)
    return (torch.randn(*shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def heavy_columns(n_cols, count, seed, stream=0):
    """`count` distinct column indices (a seeded permutation prefix), ascending."""
    g = _gen(seed, stream)
    return torch.sort(torch.randperm(n_cols, generator=g)[:count]).values


def with_heavy_columns(shape, std, factor, count, seed, stream=0):
    """N(0, std^2) with `count` fixed columns multiplied by `factor` (bf16)."""
    g = _gen(seed, stream)
    x = torch.randn(*shape, generator=g, dtype=torch.float32) * std
    cols = heavy_columns(shape[1], count, seed, stream + 7919)
    x[:, cols] *= factor
    return x.to(torch.bfloat16)


def student_t_rows(rows, cols, scale, nu, seed, stream=0):
    """Row r = scale * |T_r| * N(0,1), T_r ~ Student-t(nu) (bf16)."""
    g = _gen(seed, stream)
    z = torch.randn(rows, generator=g, dtype=torch.float64)
    chi2 = (torch.randn(rows, nu, generator=g, dtype=torch.float64) ** 2).sum(dim=1)
    t = z / torch.sqrt(chi2 / nu)
    base = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    return (base * (scale * t.abs()).to(torch.float32)[:, None]).to(torch.bfloat16)


def tiny(seed=0):
    X = with_heavy_columns((256, 512), 1.0, 50.0, 8, seed, 1)
    W = normal((512, 512), 0.02, seed, 2)
    dY = normal((256, 512), 1e-3, seed, 3)
    return X, W, dY


def quant_tensor(rows, cols, seed):
    """Quantize-sweep input: N(0,1) with ceil(1%) of the columns x30."""
    return with_heavy_columns((rows, cols), 1.0, 30.0, math.ceil(cols / 100), seed, 11)


def fwd_outctl(seed=1, M=16384, K=1024, N=4096, n_batches=4):
    """Calibration batches, the fifth batch X and W for the forward-with-OutControl case."""
    heavy = heavy_columns(K, 20, seed, 21)
    batches = []
    for b in range(n_batches + 1):
        g = _gen(seed, 100 + b)
        x = torch.randn(M, K, generator=g, dtype=torch.float32)
        x[:, heavy] *= 40.0
        batches.append(x.to(torch.bfloat16))
    W = normal((N, K), 0.02, seed, 22)
    return batches[:n_batches], batches[n_batches], W, heavy


def bwd_rht(seed=2, M=16384, N=4096, K=1024):
    dY = student_t_rows(M, N, 1e-3, 3, seed, 31)
    W = normal((N, K), 0.02, seed, 32)
    X = quant_tensor(M, K, seed)
    return dY, W, X


def layer_set_linear(name, N, K, seed=3, M=16384):
    """(X [M,K], W [N,K], dY [M,N]) for one linear of the decoder-layer set."""
    s = 40 + 10 * [n for n, _, _ in LAYER_SET].index(name)
    X = with_heavy_columns((M, K), 1.0, 30.0, math.ceil(K / 100), seed, s)
    W = normal((N, K), 0.02, seed, s + 1)
    dY = student_t_rows(M, N, 1e-3, 3, seed, s + 2)
    return X, W, dY


def cosine_lr(step, total=200, lr_max=1e-3, lr_min=1e-5):
    """Cosine-decayed learning rate of the synthetic AdamW trajectory."""
    return lr_min + 0.5 * (lr_max - lr_min) * (1.0 + math.cos(math.pi * step / total))


# ---------------------------------------------------------------------------
# Device-side generation for the benchmark (same distributions, drawn with a
# seeded CUDA generator so that multi-GB inputs appear in seconds).
# ---------------------------------------------------------------------------
OSCI_PARAMS = 22 * sum(n * k for _, n, k in LAYER_SET)       # 369,098,752 master weights


def _cuda_gen(seed, stream, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(stream))
    return g


def device_heavy_columns(shape, std, factor, count, seed, stream, device):
    g = _cuda_gen(seed, stream, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std
    cols = torch.randperm(shape[1], generator=g, device=device)[:count]
    x[:, cols] *= factor
    return x.to(torch.bfloat16)


def device_student_t_rows(rows, cols, scale, nu, seed, stream, device):
    g = _cuda_gen(seed, stream, device)
    z = torch.randn(rows, generator=g, device=device, dtype=torch.float64)
    chi2 = (torch.randn(rows, nu, generator=g, device=device, dtype=torch.float64) ** 2).sum(dim=1)
    t = (z / torch.sqrt(chi2 / nu)).abs().to(torch.float32)
    out = torch.empty(rows, cols, dtype=torch.bfloat16, device=device)
    for r0 in range(0, rows, 4096):                      # chunked: bounded fp32 temporaries
        r1 = min(rows, r0 + 4096)
        out[r0:r1] = (torch.randn(r1 - r0, cols, generator=g, device=device) * (scale * t[r0:r1, None])).to(torch.bfloat16)
    return out


def device_layer_set_linear(name, N, K, seed=3, M=16384, device="cuda"):
    """(X [M,K], W [N,K], dY [M,N]) of one linear of the layer set, on the device."""
    s = 40 + 10 * [n for n, _, _ in LAYER_SET].index(name)
    X = device_heavy_columns((M, K), 1.0, 30.0, math.ceil(K / 100), seed, s, device)
    g = _cuda_gen(seed, s + 1, device)
    W = (torch.randn(N, K, generator=g, device=device) * 0.02).to(torch.bfloat16)
    dY = device_student_t_rows(M, N, 1e-3, 3, seed, s + 2, device)
    return X, W, dY


def device_calibration_batch(K, M, heavy_count, b, seed, stream, device):
    """A calibration batch X [M,K] N(0,1) whose heavy channels (fixed per stream) are x40."""
    g = _cuda_gen(seed, stream, device)
    heavy = torch.randperm(K, generator=g, device=device)[:heavy_count]
    g2 = _cuda_gen(seed, stream + 100 + b, device)
    x = torch.randn(M, K, generator=g2, device=device)
    x[:, heavy] *= 40.0
    return x.to(torch.bfloat16)


def device_master_weights(n, seed=3, device="cuda", cols=1024):
    """OsciReset master weights w0 ~ N(0, 0.02) as [n/cols, cols] fp32."""
    g = _cuda_gen(seed, 900, device)
    w = torch.empty(n // cols, cols, dtype=torch.float32, device=device)
    for r0 in range(0, w.shape[0], 65536):
        r1 = min(w.shape[0], r0 + 65536)
        w[r0:r1].normal_(0.0, 0.02, generator=g)
    return w
