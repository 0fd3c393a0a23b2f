"""The Q4_0 linear stacks of the Voxtral Mini 4B Realtime port, run through the
library's public calls.

GeekNews (es.news.hada.io/topic?id=26595, "Arquitectura") gives the shapes:
a 26-layer decoder with hidden size 3072 and GQA 32Q/8KV (q 4096 = 32 x 128,
k and v 1024 = 8 x 128), and a 32-layer, 1280-wide causal audio encoder; on the
quantized path every one of these linears is GGUF Q4_0.  FFN widths 9216
(decoder) and 5120 (encoder) are assumptions that fit the parameter counts on
the usedby.ai post ("Bajo el capó": 3.4B LM + 0.6B encoder).

Only the linears are here: attention, norms and activations are outside the
Q4 path.  Where they would sit, the next linear reads the previous linear's
output directly (the q rows stand in for the attention output feeding wo, the
w1 rows for the gated FFN activation feeding w2), which keeps the per-layer
chain of dependent products that a real decode step has.

Layout in HBM: per decoder layer three row-concatenated matrices that share an
input -- Wqkv = [wq; wk; wv] (6144 x 3072), W13 = [w1; w3] (18432 x 3072) --
plus wo (3072 x 4096) and w2 (3072 x 9216), each a contiguous run of Q4_0 rows.
A decode step is 4 dependent products per layer (104 per step), run either as
one q4_gemv_chain launch (persistent, the weight stream never stops between
products) or as 104 q4_gemv_prefetch launches with programmatic dependent
launch between them, each prefetching the next product's weights into L2;
either is captured in a CUDA graph.
"""
from __future__ import annotations

import synth

from . import (FLAG_PDL, OP_RESIDUAL, OP_SWIGLU, Link, LinkOut, Workspace,
               interleave_gate_rows, q4_chain, q4_chain_workspace_bytes, q4_gemm, q4_gemv,
               q4_gemv_chain, q4_gemv_prefetch, q4_quantize, q4_repack)


def _quantize_rows(parts, k, device, torch):
    """Quantize several [n_i, k] fp32 matrices into one row-concatenated Q4 matrix."""
    n_total = sum(p[0] for p in parts)
    blocks = torch.empty((n_total, k // 32 * 18), dtype=torch.uint8, device=device)
    r0 = 0
    st = torch.zeros(1, dtype=torch.int32, device=device)
    for n, seed in parts:
        w = synth.torch_weights(n, k, seed=seed, device=device)
        q4_quantize(w, blocks=blocks[r0:r0 + n], status=st)
        del w
        r0 += n
    return blocks, st


class DecoderStack:
    """26 decoder layers of Q4_0 linears at one token per step."""

    HIDDEN, QDIM, KVDIM, FFN = 3072, 4096, 1024, 9216

    def __init__(self, layers: int = synth.DECODER_LAYERS, config_id: int = 2, device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.layers = layers
        H, Q, KV, F = self.HIDDEN, self.QDIM, self.KVDIM, self.FFN
        self.shapes = {"qkv": (Q + 2 * KV, H), "wo": (H, Q), "w13": (2 * F, H), "w2": (H, F)}
        self.W = []
        status = []
        for l in range(layers):
            s = lambda i: synth.seed_for(config_id, l, i)  # noqa: E731  wq..w2 = 0..6
            qkv, st1 = _quantize_rows([(Q, s(0)), (KV, s(1)), (KV, s(2))], H, self.device, torch)
            wo, st2 = _quantize_rows([(H, s(3))], Q, self.device, torch)
            w13, st3 = _quantize_rows([(F, s(4)), (F, s(5))], H, self.device, torch)
            w2, st4 = _quantize_rows([(H, s(6))], F, self.device, torch)
            self.W.append({"qkv": qkv, "wo": wo, "w13": w13, "w2": w2})
            status += [st1, st2, st3, st4]
        torch.cuda.synchronize()
        if any(int(st.item()) != 0 for st in status):
            raise RuntimeError("quantizing the decoder weights reported a device error")
        self.y_qkv = torch.empty((1, Q + 2 * KV), device=self.device)
        self.y_o = torch.empty((1, H), device=self.device)
        self.y_13 = torch.empty((1, 2 * F), device=self.device)
        self.x = torch.empty((1, H), device=self.device)
        self.ws = Workspace(self.device)
        for name, (n, k) in self.shapes.items():  # size the shared workspace once
            from . import q4_gemv_workspace_bytes
            self.ws.get(q4_gemv_workspace_bytes(n, k, 1))
        from . import q4_gemv_chain_workspace_bytes
        self.chain_ws = Workspace(self.device)
        self.chain_ws.get(q4_gemv_chain_workspace_bytes(self.links(self.x)))
        self.graphs = {}
        # the same weights in the repacked tile layout, for the fused step;
        # w1 and w3 interleaved 8 rows at a time for the gate epilogue
        self.R = []
        for layer in self.W:
            r = {name: q4_repack(w, *self.shapes[name]) for name, w in layer.items()
                 if name != "w13"}
            F = self.FFN
            w13i = interleave_gate_rows(layer["w13"][:F], layer["w13"][F:])
            r["w13"] = q4_repack(w13i, *self.shapes["w13"])
            del w13i
            self.R.append(r)
        torch.cuda.synchronize()
        self.x_fused = torch.empty((1, H), device=self.device)
        self.fused_ws = Workspace(self.device)
        self.fused_ws.get(q4_chain_workspace_bytes(self.fused_links(self.x_fused)))

    # bytes the method must move per decode step (weights once + activations)
    def weight_bytes(self) -> int:
        return sum(int(w.numel()) for layer in self.W for w in layer.values())

    def activation_bytes(self) -> int:
        per_layer = 0
        for n, k in self.shapes.values():
            per_layer += 4 * (k + n)
        return per_layer * self.layers

    def launches_per_step(self) -> int:
        return 4 * self.layers

    def _layer(self, l, x_in, stream):
        # each product prefetches the next one's weights into L2 (the last of
        # the step those of the next step's first product)
        W, (nq, h), = self.W[l], self.shapes["qkv"]
        nxt = self.W[(l + 1) % self.layers]["qkv"]
        q4_gemv_prefetch(W["qkv"], nq, h, x_in, prefetch=W["wo"], y=self.y_qkv, workspace=self.ws,
                         flags=FLAG_PDL, stream=stream)
        q4_gemv_prefetch(W["wo"], h, self.QDIM, self.y_qkv[:, :self.QDIM], prefetch=W["w13"],
                         y=self.y_o, workspace=self.ws, flags=FLAG_PDL, stream=stream)
        q4_gemv_prefetch(W["w13"], 2 * self.FFN, h, self.y_o, prefetch=W["w2"], y=self.y_13,
                         workspace=self.ws, flags=FLAG_PDL, stream=stream)
        q4_gemv_prefetch(W["w2"], h, self.FFN, self.y_13[:, :self.FFN], prefetch=nxt, y=self.x,
                         workspace=self.ws, flags=FLAG_PDL, stream=stream)

    def step_only(self, key, stream=None):
        """The products of one kind ("qkv", "wo", "w13" or "w2") of a decode step,
        one per layer, as their own chain of q4_gemv launches with programmatic
        dependent launch: timing these apart shows where a step's time goes."""
        n, k = self.shapes[key]
        src = {"qkv": self.x, "wo": self.y_qkv[:, :self.QDIM], "w13": self.y_o,
               "w2": self.y_13[:, :self.FFN]}[key]
        dst = {"qkv": self.y_qkv, "wo": self.y_o, "w13": self.y_13, "w2": self.x}[key]
        for l in range(self.layers):
            q4_gemv(self.W[l][key], n, k, src, y=dst, workspace=self.ws, flags=FLAG_PDL,
                    stream=stream)

    def capture_only(self, key, steps, stream):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.step_only(key, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(steps):
                    self.step_only(key, stream)
        return g

    def links(self, x_in):
        """The step's 104 products as chain links (W, n, k, x, y), in order."""
        H, Q, F = self.HIDDEN, self.QDIM, self.FFN
        out = []
        for l in range(self.layers):
            W = self.W[l]
            out.append((W["qkv"], Q + 2 * self.KVDIM, H, x_in if l == 0 else self.x, self.y_qkv))
            out.append((W["wo"], H, Q, self.y_qkv[:, :Q], self.y_o))
            out.append((W["w13"], 2 * F, H, self.y_o, self.y_13))
            out.append((W["w2"], H, F, self.y_13[:, :F], self.x))
        return out

    def fused_links(self, x_in, outs=None):
        """The step as one q4_chain on the repacked weights, with the decoder's
        glue fused: per layer
            qkv = Wqkv x_l
            h   = x_l + Wo q            (q = the first 4096 rows of qkv)
            g   = a * sigmoid(a) * b,  a = W1 h, b = W3 h  (in the w1/w3 product's epilogue)
            x_{l+1} = h + W2 g
        The q rows stand in for the attention output and h for its norm (both
        outside the Q4 path).  Only x_26 is written (self.x_fused) unless
        `outs` gives a buffer per link."""
        H, Q, F = self.HIDDEN, self.QDIM, self.FFN
        links = []
        for l in range(self.layers):
            R, b = self.R[l], 4 * l
            x_l = x_in if l == 0 else LinkOut(b - 1)
            y = (lambda i: outs[i]) if outs is not None else (lambda i: None)  # noqa: E731
            last = l == self.layers - 1
            links.append(Link(R["qkv"], Q + 2 * self.KVDIM, H, x_l, y=y(b)))
            links.append(Link(R["wo"], H, Q, LinkOut(b, 0), y=y(b + 1), residual=x_l,
                              ops=OP_RESIDUAL))
            links.append(Link(R["w13"], 2 * F, H, LinkOut(b + 1), y=y(b + 2), ops=OP_SWIGLU))
            links.append(Link(R["w2"], H, F, LinkOut(b + 2), residual=LinkOut(b + 1),
                              y=(self.x_fused if (last and outs is None) else y(b + 3)),
                              ops=OP_RESIDUAL))
        return links

    def fused_step(self, x_in, stream=None, outs=None):
        q4_chain(self.fused_links(x_in, outs), workspace=self.fused_ws, stream=stream)
        return self.x_fused

    def capture_fused(self, inputs, stream):
        """CUDA graph of len(inputs) consecutive fused steps."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.fused_step(inputs[0], stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for x_in in inputs:
                    self.fused_step(x_in, stream)
        return g

    def step(self, x_in, stream=None, chain: bool = False):
        """One decode step on the device: x_in [1, 3072] fp32 -> self.x [1, 3072].
        chain=True runs the 104 products as one q4_gemv_chain launch; otherwise
        one q4_gemv_prefetch launch each (programmatic dependent launch between
        them, each prefetching the next product's weights into L2)."""
        if chain:
            q4_gemv_chain(self.links(x_in), workspace=self.chain_ws, stream=stream)
            return self.x
        self._layer(0, x_in, stream)
        for l in range(1, self.layers):
            self._layer(l, self.x, stream)
        return self.x

    def capture(self, inputs, stream, chain: bool = False):
        """CUDA graph of len(inputs) consecutive steps, step i reading inputs[i]."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.step(inputs[0], stream, chain=chain)  # warm the path outside capture
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for x_in in inputs:
                    self.step(x_in, stream, chain=chain)
        return g


class EncoderStack:
    """32 encoder layers of Q4_0 linears over M audio frames (bf16 activations)."""

    DIM, FFN = 1280, 5120

    def __init__(self, frames: int, layers: int = synth.ENCODER_LAYERS, config_id: int = 4,
                 device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.layers, self.m = layers, frames
        D, F = self.DIM, self.FFN
        self.shapes = {"qkv": (3 * D, D), "out": (D, D), "up": (F, D), "down": (D, F)}
        self.W = []
        status = []
        for l in range(layers):
            s = lambda i: synth.seed_for(config_id, l, i)  # noqa: E731  qkv..down = 0..3
            qkv, a = _quantize_rows([(3 * D, s(0))], D, self.device, torch)
            out, b = _quantize_rows([(D, s(1))], D, self.device, torch)
            up, c = _quantize_rows([(F, s(2))], D, self.device, torch)
            down, d = _quantize_rows([(D, s(3))], F, self.device, torch)
            self.W.append({"qkv": qkv, "out": out, "up": up, "down": down})
            status += [a, b, c, d]
        torch.cuda.synchronize()
        if any(int(st.item()) != 0 for st in status):
            raise RuntimeError("quantizing the encoder weights reported a device error")
        bf = torch.bfloat16
        self.y_qkv = torch.empty((frames, 3 * D), dtype=bf, device=self.device)
        self.y_out = torch.empty((frames, D), dtype=bf, device=self.device)
        self.y_up = torch.empty((frames, F), dtype=bf, device=self.device)
        self.x = torch.empty((frames, D), dtype=bf, device=self.device)
        self.ws = Workspace(self.device)

    def flops_per_pass(self) -> int:
        return 2 * self.m * self.layers * sum(n * k for n, k in self.shapes.values())

    def weight_bytes(self) -> int:
        return sum(int(w.numel()) for layer in self.W for w in layer.values())

    def launches_per_pass(self) -> int:
        return 4 * self.layers

    def flops(self, frames: int) -> int:
        return 2 * frames * self.layers * sum(n * k for n, k in self.shapes.values())

    def _layer(self, l, x_in, m, stream):
        W, D, F = self.W[l], self.DIM, self.FFN
        q4_gemm(W["qkv"], 3 * D, D, x_in, Y=self.y_qkv[:m], workspace=self.ws, flags=FLAG_PDL,
                stream=stream)
        q4_gemm(W["out"], D, D, self.y_qkv[:m, :D], Y=self.y_out[:m], workspace=self.ws,
                flags=FLAG_PDL, stream=stream)
        q4_gemm(W["up"], F, D, self.y_out[:m], Y=self.y_up[:m], workspace=self.ws,
                flags=FLAG_PDL, stream=stream)
        q4_gemm(W["down"], D, F, self.y_up[:m], Y=self.x[:m], workspace=self.ws, flags=FLAG_PDL,
                stream=stream)

    def forward(self, x_in, stream=None):
        """x_in [m, 1280] bf16 with m <= frames -> self.x[:m]."""
        m = x_in.shape[0]
        self._layer(0, x_in, m, stream)
        for l in range(1, self.layers):
            self._layer(l, self.x[:m], m, stream)
        return self.x[:m]

    def capture(self, x_in, stream, passes: int = 1):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.forward(x_in, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(passes):
                    self.forward(x_in, stream)
        return g


class AdapterStack:
    """The bridge from the 1280-wide encoder to the 3072-wide decoder
    (GeekNews, "Arquitectura": "Conv with 4x downsampling -> adapter (3072
    dimensions)"), as Q4_0 linears through q4_gemm.  Shapes are assumptions
    (the pages give none): the downsampling conv has width and stride 4 over
    time, i.e. it is a linear on 4 concatenated encoder frames (5120 -> 3072),
    and the adapter is two linears 3072 -> 3072 -> 3072.  The 4-frame
    concatenation is a reshape of the row-major [frames, 1280] encoder output
    (no copy).  Activations between the linears are outside the Q4 path and
    left out, as in the other stacks."""

    def __init__(self, encoder_frames: int = synth.ADAPTER_ENCODER_FRAMES, config_id: int = 6,
                 device="cuda"):
        import torch
        if encoder_frames % 4:
            raise ValueError("encoder frames must be a multiple of 4")
        self.torch = torch
        self.device = torch.device(device)
        self.frames = encoder_frames
        self.m = encoder_frames // 4
        self.mats = synth.ADAPTER_MATS
        self.W = []
        status = []
        for idx, (_, n, k) in enumerate(self.mats):
            blocks, st = _quantize_rows([(n, synth.seed_for(config_id, 0, idx))], k, self.device,
                                        torch)
            self.W.append(blocks)
            status.append(st)
        torch.cuda.synchronize()
        if any(int(st.item()) != 0 for st in status):
            raise RuntimeError("quantizing the adapter weights reported a device error")
        bf = torch.bfloat16
        self.Y = [torch.empty((self.m, n), dtype=bf, device=self.device) for _, n, _ in self.mats]
        self.ws = Workspace(self.device)

    def flops_per_pass(self) -> int:
        return 2 * self.m * sum(n * k for _, n, k in self.mats)

    def weight_bytes(self) -> int:
        return sum(int(w.numel()) for w in self.W)

    def forward(self, X_enc, stream=None, flags: int = FLAG_PDL):
        """X_enc [frames, 1280] bf16 (row-major, contiguous) -> [frames/4, 3072] bf16."""
        x = X_enc.reshape(self.m, 4 * X_enc.shape[1])
        for W, (_, n, k), Y in zip(self.W, self.mats, self.Y):
            q4_gemm(W, n, k, x, Y=Y, workspace=self.ws, flags=flags, stream=stream)
            x = Y
        return x

    def capture(self, X_enc, stream, passes: int = 1):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            self.forward(X_enc, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(passes):
                    self.forward(X_enc, stream)
        return g


def _main(argv=None):
    """Run a few steps of a stack with no timing, for a profiler:
        python -m bit_weight_quantized_03_b300.stacks decode --layers 2 --path fused --steps 4
        python -m bit_weight_quantized_03_b300.stacks head --steps 3
    decode runs the decoder step on its per-launch (q4_gemv), chain
    (q4_gemv_chain) or fused (q4_chain, repacked) path; head runs the
    131072 x 3072 output head once per step as q4_gemv_r (repacked) and as
    q4_gemv (GGUF)."""
    import argparse

    import torch
    ap = argparse.ArgumentParser(prog="python -m bit_weight_quantized_03_b300.stacks")
    ap.add_argument("what", choices=["decode", "head"])
    ap.add_argument("--layers", type=int, default=synth.DECODER_LAYERS)
    ap.add_argument("--path", choices=["per_launch", "chain", "fused"], default="fused")
    ap.add_argument("--steps", type=int, default=3)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    if a.what == "decode":
        dec = DecoderStack(layers=a.layers, device=dev)
        x = synth.torch_activations(1, 3072, seed=synth.activation_seed(2000), device=dev)
        for _ in range(a.steps):
            if a.path == "fused":
                dec.fused_step(x)
            else:
                dec.step(x, chain=a.path == "chain")
    else:
        from . import q4_gemv_r
        V, H = synth.VOCAB, 3072
        table = torch.empty((V, H // 32 * 18), dtype=torch.uint8, device=dev)
        for r0 in range(0, V, 16384):
            w = synth.torch_weights(16384, H, seed=synth.seed_for(3, 0, r0 // 16384), device=dev)
            q4_quantize(w, blocks=table[r0:r0 + 16384])
            del w
        R = q4_repack(table, V, H)
        x = synth.torch_activations(1, H, seed=synth.activation_seed(3000), device=dev)
        y = torch.empty((1, V), device=dev)
        ws, wsr = Workspace(dev), Workspace(dev)
        for _ in range(a.steps):
            q4_gemv_r(R, V, H, x, y=y, workspace=wsr)
            q4_gemv(table, V, H, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    _main()
