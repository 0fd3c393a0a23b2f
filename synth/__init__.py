"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers: it holds none of the Q4_0 arithmetic
(no quantizing, decoding or products), so the CUDA path and the CPU oracle can
both take their inputs from it without sharing any of the method.

Shapes and distributions follow the workloads of the Voxtral Mini 4B Realtime
port described on GeekNews (es.news.hada.io/topic?id=26595, "Arquitectura":
decoder hidden 3072 with GQA 32Q/8KV over 26 layers, encoder 1280-dim over 32
layers; "Soluciones técnicas": a 1.5 GiB fp32 embedding table = 131072 x 3072).
The FFN widths (decoder 9216, encoder 5120) are assumptions that fit the
parameter counts given on the usedby.ai post ("Bajo el capó": 3.4B LM + 0.6B
audio encoder).

Weights are N(0, 0.02^2) fp32, activations N(0, 1) (fp32, or bf16 by
round-to-nearest-even), token ids uniform on [0, vocab).

Two generators:
  * numpy ``default_rng(seed)`` (PCG64) for host-side cases;
  * ``torch.Generator`` on a CUDA device (Philox) for the full-size workloads,
    which would take minutes to draw on the host.
"""
from __future__ import annotations

import numpy as np

WEIGHT_STD = 0.02

# Decoder (per layer): name -> (n_out, k_in); the order fixes the matrix index.
DECODER_HIDDEN = 3072
DECODER_LAYERS = 26
DECODER_FFN = 9216
DECODER_MATS = (("wq", 4096, 3072), ("wk", 1024, 3072), ("wv", 1024, 3072),
                ("wo", 3072, 4096), ("w1", 9216, 3072), ("w3", 9216, 3072),
                ("w2", 3072, 9216))
# Encoder (per layer)
ENCODER_DIM = 1280
ENCODER_LAYERS = 32
ENCODER_FFN = 5120
ENCODER_MATS = (("qkv", 3840, 1280), ("out", 1280, 1280), ("up", 5120, 1280),
                ("down", 1280, 5120))
ENCODER_FRAMES = (375, 1500, 3000)
VOCAB = 131072
# The bridge from the encoder to the decoder: "Conv with 4x downsampling ->
# adapter (3072 dimensions)" (GeekNews es.news.hada.io/topic?id=26595,
# "Arquitectura").  The pages give no kernel size or adapter depth; assumed
# here: the 4x downsampling is a stride-4, width-4 convolution over time (a
# linear on 4 concatenated 1280-wide encoder frames, 5120 -> 3072), then a
# two-linear adapter 3072 -> 3072 -> 3072.  1500 encoder frames (30 s) give
# 375 decoder-rate frames.
ADAPTER_ENCODER_FRAMES = 1500
ADAPTER_MATS = (("conv4x", 3072, 5120), ("adapter1", 3072, 3072), ("adapter2", 3072, 3072))


def seed_for(config: int, layer: int = 0, matrix_index: int = 0) -> int:
    """seed = 1000*config + 16*layer + matrix_index."""
    return 1000 * int(config) + 16 * int(layer) + int(matrix_index)


def activation_seed(base_seed: int, step: int = 0) -> int:
    return int(base_seed) + 500000 + int(step)


# ------------------------------------------------------------------ numpy (host)

def np_weights(n: int, k: int, seed: int, std: float = WEIGHT_STD) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, k), dtype=np.float32) * np.float32(std)).astype(np.float32)


def np_activations(m: int, k: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((m, k), dtype=np.float32)


def np_token_ids(n: int, vocab: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


# ------------------------------------------------------------------ torch (device)

def torch_weights(n: int, k: int, seed: int, device="cuda", std: float = WEIGHT_STD):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    return w.mul_(std)


def torch_activations(m: int, k: int, seed: int, device="cuda", dtype=None):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    if dtype is not None and dtype != torch.float32:
        x = x.to(dtype)  # bf16: round to nearest even
    return x


def torch_token_ids(n: int, vocab: int, seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randint(0, vocab, (n,), generator=g, device=device, dtype=torch.int32)
