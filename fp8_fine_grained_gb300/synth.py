"""Seeded synthetic inputs for the FP8 path.

This module draws random numbers and nothing else: it holds none of the
quantisation or GEMM arithmetic, so the tests can hand the same bf16 bytes to
both the CUDA library and the CPU oracle. Every tensor comes from a
``torch.Generator`` seeded per workload, on the device the caller names (the
CUDA generator is Philox; the CPU one is a Mersenne twister, so the two
devices give different but equally seeded data). Draw order inside each
recipe is fixed and written next to it.

Shapes and distributions follow the workloads of the method's setting
(DeepSeek-V3: hidden size 7168, 256 routed experts with 8 active per token);
the expert width 2048 and the MLP width 18432 are the benchmark's choices.
"""
from dataclasses import dataclass

import torch

HIDDEN = 7168


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, g, device, dtype=torch.float32):
    return torch.randn(*shape, generator=g, device=device, dtype=dtype) * std


def to_bf16(t):
    return t.to(torch.bfloat16)


# -------------------------------------------------------------- recipes ----

def tiny(seed=0, device="cpu", M=128, K=256, N=128, outlier_frac=0.01, outlier_mult=100.0):
    """Tiny fprop. Draws: X ~ N(0,1) [M,K]; W ~ N(0,0.02) [N,K]; a random
    permutation of the M*K positions, the first floor(frac*M*K) of which are
    multiplied by ``outlier_mult``."""
    g = _gen(seed, device)
    x = normal((M, K), 1.0, g, device)
    w = normal((N, K), 0.02, g, device)
    n_out = int(outlier_frac * M * K)
    idx = torch.randperm(M * K, generator=g, device=device)[:n_out]
    x.view(-1)[idx] *= outlier_mult
    return to_bf16(x), to_bf16(w)


def lognormal_channels(M, K, g, device):
    """X[m, k] = z[m, k] * c_k with z ~ N(0,1) and per-channel magnitude
    c_k = exp(N(0,1)) (log-normal, sigma 1). Draws c first, then z."""
    c = torch.exp(normal((K,), 1.0, g, device))
    z = normal((M, K), 1.0, g, device)
    return z * c


def dense(seed=0, device="cpu", M=4096, K=HIDDEN, N=HIDDEN):
    """Dense projection fprop. Draws: X (log-normal channels), then W ~ N(0,0.02) [N,K]."""
    g = _gen(seed, device)
    x = lognormal_channels(M, K, g, device)
    w = normal((N, K), 0.02, g, device)
    return to_bf16(x), to_bf16(w)


def trio(seed=0, device="cpu", M=8192, K=HIDDEN, N=18432):
    """Linear layer K -> N at M tokens, forward and both backward GEMMs.
    Draws: X (log-normal channels) [M,K]; W ~ N(0,0.02) [N,K]; dY ~ N(0,1e-3) [M,N]."""
    g = _gen(seed, device)
    x = lognormal_channels(M, K, g, device)
    w = normal((N, K), 0.02, g, device)
    dy = normal((M, N), 1e-3, g, device)
    return to_bf16(x), to_bf16(w), to_bf16(dy)


def outliers(seed=0, device="cpu", M=16384, K=HIDDEN, N=HIDDEN,
             chan_frac=0.001, chan_mult=1000.0, block_frac=0.01, block_mult=50.0):
    """Outlier-heavy fprop. Draws: X ~ N(0,1) [M,K]; W ~ N(0,0.02) [N,K];
    a permutation of the K channels, the first round(chan_frac*K) scaled by
    ``chan_mult``; a permutation of the (N/128)*(K/128) weight blocks, the
    first round(block_frac*blocks) scaled by ``block_mult``."""
    g = _gen(seed, device)
    x = normal((M, K), 1.0, g, device)
    w = normal((N, K), 0.02, g, device)
    n_ch = int(round(chan_frac * K))
    ch = torch.randperm(K, generator=g, device=device)[:n_ch]
    x[:, ch] *= chan_mult
    nbr, nbc = N // 128, K // 128
    n_bl = int(round(block_frac * nbr * nbc))
    bl = torch.randperm(nbr * nbc, generator=g, device=device)[:n_bl]
    wv = w.view(nbr, 128, nbc, 128)
    for b in bl.tolist():
        wv[b // nbc, :, b % nbc, :] *= block_mult
    return to_bf16(x), to_bf16(w), ch, bl


@dataclass
class MoEInputs:
    x: torch.Tensor            # bf16 [T, K]
    w: torch.Tensor            # bf16 [E, N, K]
    row_index: torch.Tensor    # int32 [T*topk]: token of each expert row, grouped by expert
    expert_offsets: torch.Tensor  # int32 [E+1]
    counts: torch.Tensor       # int64 [E]
    topk_ids: torch.Tensor = None  # int32 [T, topk]: each token's experts, best first
    gates: torch.Tensor = None     # float32 [T, topk]: softmax of the chosen experts' logits (no bias)


def route_topk(logits, bias, topk):
    """Top-k experts per token of (logits + bias), ties to the lower expert
    index; returns (row_index, expert_offsets, counts) with rows grouped by
    expert ascending and, within an expert, by token ascending. Softmax is
    monotone, so ranking logits + bias equals ranking its softmax."""
    T, E = logits.shape
    score = (logits + bias).float()
    # stable sort of -score keeps the lower index first among equal scores
    order = torch.sort(-score, dim=1, stable=True).indices[:, :topk]
    tok = torch.arange(T, device=logits.device).unsqueeze(1).expand(T, topk).reshape(-1)
    exp = order.reshape(-1)
    key = exp.to(torch.int64) * T + tok
    perm = torch.sort(key, stable=True).indices
    row_index = tok[perm].to(torch.int32)
    counts = torch.bincount(exp, minlength=E)
    off = torch.zeros(E + 1, dtype=torch.int64, device=logits.device)
    off[1:] = torch.cumsum(counts, 0)
    return row_index, off.to(torch.int32), counts


def moe(seed=0, device="cpu", T=4096, K=HIDDEN, N=2048, E=256, topk=8, zipf_s=1.1,
        make_weights=True):
    """MoE expert GEMM inputs. Draws: X ~ N(0,1) [T,K]; logits ~ N(0,1) [T,E];
    a permutation r of 1..E (expert popularity ranks); W ~ N(0,0.02) [E,N,K].
    Per-expert bias b_e = -zipf_s * ln(r_e), i.e. Zipf(zipf_s) popularity."""
    g = _gen(seed, device)
    x = normal((T, K), 1.0, g, device)
    logits = normal((T, E), 1.0, g, device)
    ranks = torch.randperm(E, generator=g, device=device).to(torch.float32) + 1.0
    bias = -zipf_s * torch.log(ranks)
    w = normal((E, N, K), 0.02, g, device) if make_weights else None
    row_index, off, counts = route_topk(logits, bias, topk)
    # the combine's gate weights: the chosen experts ranked as route_topk
    # ranks them, weighted by the softmax of their own logits (the per-expert
    # bias only enters the choice); no further random draws
    ids = torch.sort(-(logits + bias).float(), dim=1, stable=True).indices[:, :topk]
    gates = torch.softmax(torch.gather(logits.float(), 1, ids), dim=1)
    return MoEInputs(to_bf16(x), to_bf16(w) if w is not None else None, row_index, off, counts,
                     ids.to(torch.int32).contiguous(), gates.contiguous())


def bf16_bits(t):
    """bf16 tensor -> numpy uint16 bit patterns on the host (for the oracle)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
