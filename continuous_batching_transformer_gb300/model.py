"""Device-side model and engine handles for the synthetic workloads.

``DeviceWeights`` lays a ModelShape's seeded weights out in the engine's format (fused
[q;k;v] and [gate;up] matrices, bf16 or 4-bit affine) directly in device memory, drawing
every value with the shared counter-based generator (``synth``), so the oracle sees the
same numbers in its own layout.  ``Engine`` owns a KV arena tensor and an engine handle.
"""
from __future__ import annotations

import ctypes

import torch

import synth
from synth.recipes import ModelShape

from . import binding as B


def config_struct(shape: ModelShape) -> B.ModelConfig:
    return B.ModelConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                         shape.head_dim, shape.d_ff, shape.vocab, shape.rms_eps, shape.rope_theta,
                         B.WEIGHTS_BF16 if shape.weight_format == "bf16" else B.WEIGHTS_AFFINE4,
                         shape.group_size)


class DeviceWeights:
    def __init__(self, shape: ModelShape, device="cuda"):
        self.shape = s = shape
        self.device = torch.device(device)
        self.tensors = []
        self.fmt = s.weight_format
        seed, sig = s.weight_seed, s.weight_sigma
        d, qd, kvd, F, V = s.d_model, s.q_dim, s.kv_dim, s.d_ff, s.vocab
        stream = torch.cuda.current_stream(self.device).cuda_stream

        def bf16_tensor(rows, cols, parts):
            """parts: [(stream_id, n_rows)] filled back to back."""
            t = torch.empty((rows, cols), dtype=torch.bfloat16, device=self.device)
            off = 0
            for st, nr in parts:
                synth.dev_normal_bf16(t.data_ptr() + off * cols * 2, nr * cols, seed, st,
                                      sigma=sig, cuda_stream=stream)
                off += nr
            return t

        def linear(rows, cols, parts):
            w = bf16_tensor(rows, cols, parts)
            if self.fmt == "bf16":
                self.tensors.append(w)
                return B.Linear(w.data_ptr(), None, None)
            G = s.group_size
            packed = torch.empty((rows, cols // 8), dtype=torch.int32, device=self.device)
            scales = torch.empty((rows, cols // G), dtype=torch.bfloat16, device=self.device)
            biases = torch.empty((rows, cols // G), dtype=torch.bfloat16, device=self.device)
            B.quantize_affine4(w.data_ptr(), rows, cols, G, packed.data_ptr(), scales.data_ptr(),
                               biases.data_ptr(), stream)
            torch.cuda.current_stream(self.device).synchronize()
            del w
            self.tensors += [packed, scales, biases]
            return B.Linear(packed.data_ptr(), scales.data_ptr(), biases.data_ptr())

        def gain(layer, kind):
            t = torch.empty(d, dtype=torch.bfloat16, device=self.device)
            synth.dev_normal_bf16(t.data_ptr(), d, seed, synth.stream_weight(layer, kind),
                                  mean=1.0, sigma=s.gain_sigma, cuda_stream=stream)
            self.tensors.append(t)
            return t.data_ptr()

        sw = synth.stream_weight
        self.embed = bf16_tensor(V, d, [(sw(-1, synth.EMBED), V)])
        self.tensors.append(self.embed)
        self.lm_head = linear(V, d, [(sw(-1, synth.LM_HEAD), V)])
        self.final_norm = gain(-1, synth.FINAL_NORM)
        self.layers = (B.LayerWeights * s.n_layers)()
        for l in range(s.n_layers):
            self.layers[l] = B.LayerWeights(
                linear(qd + 2 * kvd, d, [(sw(l, synth.WQ), qd), (sw(l, synth.WK), kvd),
                                         (sw(l, synth.WV), kvd)]),
                linear(d, qd, [(sw(l, synth.WO), d)]),
                linear(2 * F, d, [(sw(l, synth.WG), F), (sw(l, synth.WU), F)]),
                linear(d, F, [(sw(l, synth.WD), d)]),
                gain(l, synth.ATTN_NORM), gain(l, synth.FFN_NORM))
        torch.cuda.current_stream(self.device).synchronize()
        self.struct = B.Weights(self.embed.data_ptr(), self.lm_head, self.final_norm,
                                ctypes.cast(self.layers, ctypes.POINTER(B.LayerWeights)))
        self.cfg = config_struct(s)


class Engine:
    """An engine over DeviceWeights with its own KV arena (a torch tensor)."""

    def __init__(self, weights: DeviceWeights, arena_bytes: int, max_batch: int,
                 max_prefill_tokens: int, stream: torch.cuda.Stream | None = None,
                 page_tokens: int = 0, kv_bits: int = 16):
        """page_tokens > 0 (a multiple of 128): paged KV, slabs take pages of that many
        positions from the arena as they grow.  kv_bits = 8 or 4: affine KV of that many bits."""
        self.weights = weights
        self.shape = weights.shape
        self.arena = torch.empty(arena_bytes, dtype=torch.uint8, device=weights.device)
        self.stream = stream or torch.cuda.current_stream(weights.device)
        params = B.EngineParams(self.arena.data_ptr(), arena_bytes, max_batch, max_prefill_tokens,
                                self.stream.cuda_stream, page_tokens, kv_bits)
        self.page_tokens = page_tokens
        self.kv_bits = kv_bits
        self.handle = B.engine_create(weights.cfg, weights.struct, params)
        self.max_batch = max_batch
        self.max_prefill_tokens = max_prefill_tokens

    def close(self):
        if self.handle:
            B.engine_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # thin forwards to the C ABI
    def kv_slab_alloc(self, capacity: int) -> int:
        return B.kv_slab_alloc(self.handle, capacity)

    def kv_slab_free(self, slab: int) -> None:
        B.kv_slab_free(self.handle, slab)

    def retire(self, slabs) -> None:
        B.retire(self.handle, list(slabs))

    def position(self, slab: int) -> int:
        return B.kv_slab_position(self.handle, slab)

    def import_kv(self, slab: int, k: torch.Tensor, v: torch.Tensor, n_tokens: int) -> None:
        on_host = k.device.type == "cpu"
        B.kv_slab_import(self.handle, slab, k.data_ptr(), v.data_ptr(), n_tokens, on_host)

    def copy_prefix(self, src: int, dst: int, n_tokens: int) -> None:
        """dst takes positions [0, n_tokens) of src (a shared prompt prefix computed once)."""
        B.kv_slab_copy_prefix(self.handle, src, dst, n_tokens)

    def share_prefix(self, src: int, dst: int, n_tokens: int) -> None:
        """dst (at position 0) takes positions [0, n_tokens) of src by reference: on a paged
        engine the pages are shared and copied only when one of the slabs writes into one."""
        B.kv_slab_share_prefix(self.handle, src, dst, n_tokens)

    def export_kv(self, slab: int, k: torch.Tensor, v: torch.Tensor, n_tokens: int) -> None:
        on_host = k.device.type == "cpu"
        B.kv_slab_export(self.handle, slab, k.data_ptr(), v.data_ptr(), n_tokens, on_host)

    def prefill_segmented(self, slabs, seg_lens, tokens: torch.Tensor,
                          logits: torch.Tensor | None = None, next_tokens: torch.Tensor | None = None):
        B.prefill_segmented(self.handle, list(slabs), list(seg_lens), tokens.data_ptr(),
                            logits.data_ptr() if logits is not None else None,
                            next_tokens.data_ptr() if next_tokens is not None else None)

    def decode_step_batch(self, slabs, last_tokens: torch.Tensor,
                          logits: torch.Tensor | None = None, next_tokens: torch.Tensor | None = None):
        B.decode_step_batch(self.handle, list(slabs), last_tokens.data_ptr(),
                            logits.data_ptr() if logits is not None else None,
                            next_tokens.data_ptr() if next_tokens is not None else None)

    def device_error(self):
        return B.last_device_error(self.handle)

    def stats(self) -> B.Stats:
        return B.engine_stats(self.handle)

    def fill_synthetic_kv(self, slab: int, row: int, n_tokens: int, seed: int) -> None:
        """Load positions [0, n_tokens) of a slab with the seeded synthetic KV of `row`
        (the same draws the oracle's KVCache.fill_synthetic uses)."""
        s = self.shape
        dims = (s.n_layers, s.n_kv_heads, n_tokens, s.head_dim)
        st = self.stream.cuda_stream
        k = torch.empty(dims, dtype=torch.bfloat16, device=self.weights.device)
        v = torch.empty(dims, dtype=torch.bfloat16, device=self.weights.device)
        synth.dev_kv(k.data_ptr(), row, 0, s.n_layers, s.n_kv_heads, n_tokens, s.head_dim, seed,
                     s.kv_sigma, st)
        synth.dev_kv(v.data_ptr(), row, 1, s.n_layers, s.n_kv_heads, n_tokens, s.head_dim, seed,
                     s.kv_sigma, st)
        self.import_kv(slab, k, v, n_tokens)
        self.stream.synchronize()
