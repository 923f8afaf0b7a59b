"""The verify pass of a 27B-shaped dense 4-bit model on one GPU, assembled from libsvd calls.

A pass is 64 layers x 4 fused verify-linear products (q|k|v, o, gate|up, down; every matrix read
from HBM once and applied to the C = K+1 window columns), run as one persistent chain launch, then the lm_head over all C positions
with the production sampler, then the acceptance of the K drafts -- "100 tokens per second ..."
(section "How speculative decoding gets past a per-token wall") and the HN thread's account of
running every window position through each layer with one weight read.  The stack is recorded
once into a CUDA graph; a second graph holds lm_head, sampler and acceptance.

The activations of every linear are independent synthetic N(0, 1) draws (there is no real model:
attention, norms and activations between the GEMMs are out of scope), so each launch reads its
own resident X and writes its own Y, in the stream order of the real dependency chain.
"""
from __future__ import annotations

import torch

from . import roofline, svd, synth

# Drafter noise giving alpha ~ 0.5 under the production sampler; computed by the oracle-only
# script oracle/calibrate_sigma.py (stored in tests/golden/drafter_sigma.json).
DRAFTER_SIGMA = 1.2053885962814093


class Linear:
    """One 4-bit matrix resident in the native layout, with its input and output buffers."""

    def __init__(self, in_f: int, out_f: int, C: int, seed: int, device, keep_canonical=False):
        codes, scales = synth.qweight_torch(out_f, in_f, seed, device)
        cb, sb = svd.svd_native_sizes(in_f, out_f)
        self.codes = torch.empty(cb, dtype=torch.uint8, device=device)
        self.scales = torch.empty(sb, dtype=torch.uint8, device=device)
        svd.svd_repack_weights(svd.QWeight(codes, scales, in_f, out_f, svd.SVD_LAYOUT_CANONICAL),
                               self.codes, self.scales)
        self.W = svd.QWeight(self.codes, self.scales, in_f, out_f, svd.SVD_LAYOUT_NATIVE)
        self.canonical = (codes, scales) if keep_canonical else None
        self.in_f, self.out_f, self.C = in_f, out_f, C
        self.X = synth.activations_torch(C, in_f, seed + 7919, device)
        self.Y = torch.empty((C, out_f), dtype=torch.float32, device=device)


class VerifyPass:
    def __init__(self, layers: int = synth.LAYERS, C: int = 4, seed: int = 0, device="cuda",
                 head: bool = True, accept: bool = True, sampler: svd.Sampler | None = None,
                 pdl: bool = True, keep_canonical: bool = False, gemms=synth.LAYER_GEMMS,
                 chain: bool = True):
        self.device = torch.device(device)
        self.C, self.layers, self.pdl, self.chain = C, layers, pdl, chain
        self.gemms = tuple(gemms)
        self.sampler = sampler or svd.Sampler(0.6, 0.95, 0.05)
        self.linears = []
        for l in range(layers):
            for g, (i, o) in enumerate(self.gemms):
                self.linears.append(Linear(i, o, C, seed * 100003 + 1000 * l + g, self.device,
                                           keep_canonical))
        self.ops = [(lin.W, lin.X, lin.Y) for lin in self.linears]
        ws = max(max(svd.svd_verify_linear_workspace_bytes(i, o, C) for i, o in self.gemms),
                 svd.svd_verify_chain_workspace_bytes(self.ops, C))
        self.ws = torch.zeros(ws, dtype=torch.uint8, device=self.device)
        self.head = head
        self.k = C - 1
        if head:
            self.lm = Linear(synth.HIDDEN, synth.VOCAB, C, seed * 100003 + 999_999, self.device,
                             keep_canonical)
            V = synth.VOCAB
            self.V = V
            self.probs = torch.empty((C, V), dtype=torch.float32, device=self.device)
            self.argmax = torch.empty(C, dtype=torch.int32, device=self.device)
            self.head_ws = torch.zeros(svd.svd_lm_head_workspace_bytes(synth.HIDDEN, V, C),
                                       dtype=torch.uint8, device=self.device)
        self.accept = accept and head and self.k >= 1
        if self.accept:
            self._setup_drafter(seed)
        self.g_stack = self.g_tail = None
        torch.cuda.synchronize()

    # -- the drafter of the window (untimed set-up) -----------------------------------------
    def _setup_drafter(self, seed: int):
        k, V = self.k, self.V
        self.enqueue_tail(with_accept=False)
        gen = torch.Generator(device=self.device)
        gen.manual_seed(seed + 31337)
        noise = torch.empty((k, V), dtype=torch.float32, device=self.device)
        noise.normal_(0.0, DRAFTER_SIGMA, generator=gen)
        self.q_logits = (self.lm.Y[:k] + noise).contiguous()
        self.q = torch.empty((k, V), dtype=torch.float32, device=self.device)
        qam = torch.empty(k, dtype=torch.int32, device=self.device)
        qws = torch.zeros(svd.svd_sampler_workspace_bytes(k, V), dtype=torch.uint8,
                          device=self.device)
        svd.svd_sampler_probs(self.q_logits, k, V, self.sampler, self.q, qam, qws)
        self.draft = torch.multinomial(self.q, 1, generator=gen).to(torch.int32).view(1, k)
        self.tokens = torch.empty((1, k + 1), dtype=torch.int32, device=self.device)
        self.n_emitted = torch.empty(1, dtype=torch.int32, device=self.device)
        self.status = torch.empty(1, dtype=torch.int32, device=self.device)
        self.seed = seed

    # -- enqueueing -------------------------------------------------------------------------
    def enqueue_stack(self, stream=None):
        """The layer stack: one persistent cooperative chain launch (default), or one launch per
        matrix with programmatic dependent launch."""
        if self.chain:
            svd.svd_verify_chain(self.ops, self.C, self.ws, stream=stream)
            return
        flags = svd.SVD_F_PDL if self.pdl else 0
        for lin in self.linears:
            svd.svd_verify_linear(lin.W, lin.X, self.C, lin.Y, self.ws, flags=flags, stream=stream)

    def enqueue_tail(self, stream=None, with_accept=True):
        if not self.head:
            return
        svd.svd_lm_head_softmax(self.lm.W, self.lm.X, self.C, self.sampler, self.lm.Y, self.probs,
                                self.argmax, self.head_ws, stream=stream)
        if with_accept and self.accept:
            svd.svd_accept(self.probs, self.draft, 1, self.k, self.V, self.tokens, self.n_emitted,
                           self.status, q=self.q, seed=self.seed, stream=stream)

    def capture(self):
        """Record the stack and the tail into two CUDA graphs (after one eager warm-up)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.enqueue_stack(s)
            self.enqueue_tail(s)
            s.synchronize()
            svd.svd_graph_begin(s)
            self.enqueue_stack(s)
            self.g_stack = svd.svd_graph_end(s)
            if self.head:
                svd.svd_graph_begin(s)
                self.enqueue_tail(s)
                self.g_tail = svd.svd_graph_end(s)
        s.synchronize()
        return self

    def launch(self, stream=None, ev_mid=None):
        self.g_stack.launch(stream)
        if ev_mid is not None:
            ev_mid.record(stream)
        if self.g_tail is not None:
            self.g_tail.launch(stream)

    # -- accounting -------------------------------------------------------------------------
    def stack_bytes(self) -> int:
        return self.layers * sum(roofline.linear_bytes(i, o, self.C) for i, o in self.gemms)

    def stack_flops(self) -> int:
        return self.layers * sum(roofline.linear_flops(i, o, self.C) for i, o in self.gemms)

    def pass_bytes(self) -> int:
        b = self.stack_bytes()
        if self.head:
            b += roofline.head_bytes(self.C)
        if self.accept:
            b += roofline.accept_bytes_per_window(self.V, self.k, True)
        return b

    def inputs(self):
        """What a verify pass receives from the host (copied host -> device in the end-to-end
        measurement): the first layer's input (the embedded window, C x 5120 bf16), the drafter's
        distributions q and the drafts.  The other layers' activations stand for what the model
        computes on the device from the previous layer's output, so they stay resident."""
        t = [self.linears[0].X]
        if self.accept:
            t += [self.q, self.draft]
        return t

    def outputs(self):
        if self.accept:
            return [self.tokens, self.n_emitted, self.status]
        if self.head:
            return [self.argmax]
        return [self.linears[-1].Y]


class ColumnsView:
    """The resident weights of a VerifyPass applied to a window of another width C: new
    activations and outputs, the same 4-bit matrices, the stack as one chain launch (for the
    sweep over window widths without re-creating 12 GB of weights)."""

    def __init__(self, vp: VerifyPass, C: int, seed: int = 0, flags: int = 0):
        self.vp, self.C, self.flags = vp, C, flags
        dev = vp.device
        self.X = [synth.activations_torch(C, lin.in_f, seed * 100003 + n, dev)
                  for n, lin in enumerate(vp.linears)]
        self.Y = [torch.empty((C, lin.out_f), dtype=torch.float32, device=dev) for lin in vp.linears]
        self.ops = [(lin.W, x, y) for lin, x, y in zip(vp.linears, self.X, self.Y)]
        self.ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(self.ops, C), dtype=torch.uint8,
                              device=dev)
        self.graph = None

    def enqueue(self, stream=None):
        svd.svd_verify_chain(self.ops, self.C, self.ws, flags=self.flags, stream=stream)

    def capture(self):
        s = torch.cuda.Stream(device=self.vp.device)
        s.wait_stream(torch.cuda.current_stream(self.vp.device))
        with torch.cuda.stream(s):
            self.enqueue(s)
            s.synchronize()
            svd.svd_graph_begin(s)
            self.enqueue(s)
            self.graph = svd.svd_graph_end(s)
        s.synchronize()
        return self

    def launch(self, stream=None):
        self.graph.launch(stream)

    def stack_bytes(self) -> int:
        return self.vp.layers * sum(roofline.linear_bytes(i, o, self.C) for i, o in self.vp.gemms)


class Q4kStack:
    """The 27B-shaped stack in the pages' own checkpoint format: every matrix drawn as Q4_K
    super-blocks ("100 tokens per second ...", "The wall": UD-Q4_K_XL / Q4_K_M), repacked once
    into the Q4_K native layout, and the 256 products run as one chain launch recorded in a CUDA
    graph -- the same pass as VerifyPass's stack with the K-quant weights in place of the
    symmetric 4.5-bit format (the same 144 bytes per 256 weights)."""

    def __init__(self, layers: int = synth.LAYERS, C: int = 4, seed: int = 0, device="cuda",
                 gemms=synth.LAYER_GEMMS):
        self.device = torch.device(device)
        self.C, self.layers, self.gemms = C, layers, tuple(gemms)
        self.ops, self._keep = [], []
        for l in range(layers):
            for g, (i, o) in enumerate(self.gemms):
                raw = synth.q4k_blocks_torch(o, i, seed * 100003 + 1000 * l + g, self.device)
                cb, hb = svd.svd_q4k_native_sizes(i, o)
                codes = torch.empty(cb, dtype=torch.uint8, device=self.device)
                hdr = torch.empty(hb, dtype=torch.uint8, device=self.device)
                svd.svd_repack_weights(svd.QWeight(raw, None, i, o, svd.SVD_LAYOUT_Q4K), codes, hdr)
                del raw
                W = svd.QWeight(codes, hdr, i, o, svd.SVD_LAYOUT_Q4K_NATIVE)
                X = synth.activations_torch(C, i, seed * 100003 + 7919 + 1000 * l + g, self.device)
                Y = torch.empty((C, o), dtype=torch.float32, device=self.device)
                self.ops.append((W, X, Y))
                self._keep.append((codes, hdr))
        self.ws = torch.zeros(svd.svd_verify_chain_workspace_bytes(self.ops, C), dtype=torch.uint8,
                              device=self.device)
        self.graph = None
        torch.cuda.synchronize(self.device)

    def enqueue(self, stream=None):
        svd.svd_verify_chain(self.ops, self.C, self.ws, stream=stream)

    def capture(self):
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.enqueue(s)
            s.synchronize()
            svd.svd_graph_begin(s)
            self.enqueue(s)
            self.graph = svd.svd_graph_end(s)
        s.synchronize()
        return self

    def launch(self, stream=None):
        self.graph.launch(stream)

    def stack_bytes(self) -> int:
        return self.layers * sum(roofline.q4k_linear_bytes(i, o, self.C) for i, o in self.gemms)


class KvPass:
    """The resident weights of a VerifyPass with every layer's KV cache in its place, between the
    layer's q|k|v product and its o product: svd_kv_attention_append -- the window's keys and
    values (the k and v columns of the q|k|v output) quantised to q8_0/q4_0 at the window's cache
    positions, then the window's C queries attending over the layer's own cache (40 query heads
    over 8 kv heads of dimension 128, the window at positions context - C .. context - 1).  The
    matrices between two attention steps (o, gate|up and down of one layer with q|k|v of the
    next) form one chain launch, so a pass is 65 chain launches and 64 append + attention steps,
    recorded into one CUDA graph.  "Decode is memory-bound ..." ("The ceiling"): at long context
    the KV cache joins the weights on every pass.  Queries and attention outputs are synthetic
    buffers of their own, like the stack's other activations; the stream order is the model's."""

    def __init__(self, vp: VerifyPass, context: int, seed: int = 0, append: bool = True):
        self.vp, self.context, self.append = vp, context, append
        dev, C = vp.device, vp.C
        Hq, Hkv, D = synth.N_Q_HEADS, synth.N_KV_HEADS, synth.HEAD_DIM
        self.Hq, self.Hkv, self.D = Hq, Hkv, D
        kc, ks, vc, vs = synth.kv_cache_torch(Hkv, context, D, seed, dev)
        nbytes = svd.svd_kv_cache_bytes(Hkv, context)
        self.caches = []
        for _ in range(vp.layers):
            cache = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            svd.svd_kv_repack(kc, ks, vc, vs, Hkv, context, 0, context, cache, context)
            self.caches.append(cache)
        del kc, ks, vc, vs
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 17)
        self.q = torch.randn((C, Hq, D), generator=g, device=dev).to(torch.bfloat16)
        self.o = torch.empty((C, Hq, D), dtype=torch.float32, device=dev)
        self.att_ws = torch.zeros(svd.svd_kv_attention_workspace_bytes(Hq, Hkv, C),
                                  dtype=torch.uint8, device=dev)
        # Chain segments between the attention steps: q|k|v of layer 0; then o, gate|up, down of
        # layer l with q|k|v of layer l + 1; the last layer's o, gate|up, down alone.
        n = len(vp.gemms)
        self.segments = [vp.ops[0:1]]
        for l in range(vp.layers):
            self.segments.append(vp.ops[n * l + 1:n * (l + 1) + 1])
        self.graph = None
        torch.cuda.synchronize()

    def enqueue(self, stream=None):
        vp = self.vp
        n = len(vp.gemms)
        for l in range(vp.layers):
            svd.svd_verify_chain(self.segments[l], vp.C, vp.ws, stream=stream)
            if self.append:
                # the window's keys and values, columns 5120.. and 6144.. of the q|k|v output,
                # quantised into the cache by the attention kernel itself
                y = vp.linears[n * l].Y
                base, row = y.data_ptr(), y.shape[1]
                svd.svd_kv_attention_append(
                    self.q, base + 4 * synth.HIDDEN, base + 4 * (synth.HIDDEN + self.Hkv * self.D),
                    row, self.caches[l], self.context, self.Hq, self.Hkv, self.context - vp.C,
                    vp.C, 1.0 / self.D ** 0.5, self.o, self.att_ws, stream=stream)
            else:
                svd.svd_kv_attention(self.q, self.caches[l], self.context, self.Hq, self.Hkv,
                                     self.context - vp.C, vp.C, 1.0 / self.D ** 0.5, self.o,
                                     self.att_ws, stream=stream)
        svd.svd_verify_chain(self.segments[vp.layers], vp.C, vp.ws, stream=stream)

    def capture(self):
        s = torch.cuda.Stream(device=self.vp.device)
        s.wait_stream(torch.cuda.current_stream(self.vp.device))
        with torch.cuda.stream(s):
            self.enqueue(s)
            s.synchronize()
            svd.svd_graph_begin(s)
            self.enqueue(s)
            self.graph = svd.svd_graph_end(s)
        s.synchronize()
        return self

    def launch(self, stream=None):
        self.graph.launch(stream)

    def kv_bytes(self) -> int:
        return self.vp.layers * (self.Hkv * -(-self.context // 16) * svd.SVD_KV_UNIT_BYTES
                                 + self.vp.C * self.Hq * self.D * (2 + 4))

    def launches(self) -> int:
        return len(self.segments) + 2 * self.vp.layers
