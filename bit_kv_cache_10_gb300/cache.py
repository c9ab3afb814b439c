"""Torch-facing wrapper of the C ABI: a packed KV cache whose buffers are torch
tensors on one CUDA device.  Argument marshalling only -- every step of the
quantize, decode and dequantize paths runs in the CUDA library.

Shapes follow the ``TurboQuantKVCache`` of the MLX-VLM deep-dive ("The
TurboQuantKVCache Class"): packed uint32 words per token plus a float32 norm,
with the (batch, KV head, position) shape kept so that slices stay cheap.
"""
from __future__ import annotations

import torch

from . import native as N


# Raw handle of a device's current stream without building a Stream object (a
# tenth of the host time of torch.cuda.current_stream); the public call where
# this torch build lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(device) -> int:
    if _raw_stream is not None and device.index is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


class TurboQuantKVCache:
    """Packed K/V cache of one attention layer.

    ``bits`` may be fractional (K gets floor, V gets ceil), a (k_bits,
    v_bits) pair, or "int8" for the per-token INT8 absmax mode (int8 K and V
    codes, the norms buffers holding the absmax scales; no rotation);
    ``k_fp16=True`` keeps K in fp16 (the asym modes);
    ``hot_window`` > 0 keeps the newest V tokens in an fp16 ring;
    ``sparse_v_threshold`` > 0 lets decode skip the V rows of (token, head)
    pairs whose softmax weight is below it (0 decodes densely);
    ``block_size`` > 0 selects the paged layout: K/V and norms live in pools of
    ``num_blocks`` blocks (default: enough for every sequence at full
    capacity) and ``block_table`` [B, capacity / block_size] (int32, on the
    device, initially sequence b -> blocks b * n .. b * n + n - 1) maps each
    sequence's positions to blocks; it may be rewritten between calls.
    """

    def __init__(self, batch: int, num_kv_heads: int, num_q_heads: int, capacity: int, bits=3.5,
                 head_dim: int = 128, k_fp16: bool = False, hot_window: int = 0, seed: int = 0, layer: int = 0,
                 device="cuda", sparse_v_threshold: float = 0.0, block_size: int = 0, num_blocks=None):
        int8 = isinstance(bits, str)
        if int8:
            if bits != "int8" or k_fp16:
                raise ValueError('bits must be a number, a (k_bits, v_bits) pair or "int8" (with packed K)')
            k_bits, v_bits = 8, 8
        elif isinstance(bits, tuple):
            k_bits, v_bits = bits
        else:
            k_bits, v_bits = N.tq_split_bits(float(bits))
        self.int8 = int8
        mode = N.TQ_KV_INT8 if int8 else N.TQ_K_FP16 if k_fp16 else N.TQ_K_PACKED
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.desc = N.tq_cache_desc_init(batch, num_kv_heads, num_q_heads, head_dim, capacity,
                                         mode, 0 if k_fp16 else k_bits, v_bits,
                                         hot_window, seed, layer)
        d = self.desc
        self.batch, self.num_kv_heads, self.num_q_heads = batch, num_kv_heads, num_q_heads
        self.head_dim, self.capacity, self.hot_window = head_dim, capacity, hot_window
        self.k_bits = 16 if k_fp16 else k_bits
        self.v_bits = v_bits
        if block_size > 0:
            if capacity % block_size:
                raise ValueError("capacity must be a multiple of block_size")
            max_blocks = capacity // block_size
            num_blocks = batch * max_blocks if num_blocks is None else int(num_blocks)
            self.block_table = (torch.arange(batch * max_blocks, dtype=torch.int32, device=self.device)
                                .view(batch, max_blocks) % num_blocks).contiguous()
            N.tq_cache_desc_set_paged(self.desc, block_size, max_blocks, num_blocks, self.block_table.data_ptr())
            shape = (num_blocks, num_kv_heads, block_size)  # pools
        else:
            self.block_table = None
            shape = (batch, num_kv_heads, capacity)
        self.block_size, self.num_blocks = block_size, (num_blocks if block_size > 0 else 0)
        if k_fp16:
            self.k_cache = torch.zeros(*shape, head_dim, dtype=torch.float16, device=self.device)
            self.k_norms = None
        else:
            self.k_cache = torch.zeros(*shape, head_dim * k_bits // 32, dtype=torch.int32, device=self.device)
            self.k_norms = torch.zeros(*shape, dtype=torch.float32, device=self.device)
        self.v_cache = torch.zeros(*shape, head_dim * v_bits // 32, dtype=torch.int32, device=self.device)
        self.v_norms = torch.zeros(*shape, dtype=torch.float32, device=self.device)
        self.v_hot = (torch.zeros(batch, num_kv_heads, hot_window, head_dim, dtype=torch.float16, device=self.device)
                      if hot_window > 0 else None)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        d.k_cache = self.k_cache.data_ptr()
        d.k_norms = self.k_norms.data_ptr() if self.k_norms is not None else None
        d.v_cache = self.v_cache.data_ptr()
        d.v_norms = self.v_norms.data_ptr()
        d.v_hot = self.v_hot.data_ptr() if self.v_hot is not None else None
        d.d_status = self.status.data_ptr()
        d.sparse_v_threshold = float(sparse_v_threshold)
        self._workspace = None

    # -- update ---------------------------------------------------------------
    def append(self, k: torch.Tensor, v: torch.Tensor, start_pos: torch.Tensor,
               num_new: torch.Tensor | None = None) -> None:
        """Quantize and store fp16 K/V [B, Hkv, n_new, d] at positions start_pos[b] + t.

        ``k`` and ``v`` must have the same strides with a contiguous last
        dimension; ``start_pos`` is an int32 device tensor [B]; the optional
        int32 ``num_new`` [B] limits sequence b to its first num_new[b] rows."""
        if k.dtype != torch.float16 or v.dtype != torch.float16 or k.shape != v.shape or k.stride() != v.stride():
            raise ValueError("k and v must be fp16 tensors of equal shape and strides")
        if k.dim() != 4 or k.stride(3) != 1 or k.device != self.device:
            raise ValueError("k/v must be [B, Hkv, n_new, d] on the cache device with contiguous d")
        if start_pos.dtype != torch.int32 or start_pos.device != self.device or not start_pos.is_contiguous():
            raise ValueError("start_pos must be a contiguous int32 tensor on the cache device")
        if num_new is not None and (num_new.dtype != torch.int32 or num_new.device != self.device
                                    or not num_new.is_contiguous()):
            raise ValueError("num_new must be a contiguous int32 tensor on the cache device")
        N.tq_quantize_append(self.desc, k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2),
                             k.shape[2], start_pos.data_ptr(), num_new.data_ptr() if num_new is not None else None,
                             _stream_handle(self.device))

    # -- decode ---------------------------------------------------------------
    def workspace_bytes(self, max_seq_len: int) -> int:
        return N.tq_decode_workspace_bytes(self.desc, max_seq_len)

    def decode(self, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None) -> torch.Tensor:
        """Attention of fp16 queries [B, Hq, d] over the cache; returns float32 [B, Hq, d]."""
        if q.dtype != torch.float16 or not q.is_contiguous() or q.shape != (self.batch, self.num_q_heads, self.head_dim):
            raise ValueError("q must be a contiguous fp16 tensor [B, Hq, d]")
        if seq_lens.dtype != torch.int32 or seq_lens.device != self.device or not seq_lens.is_contiguous():
            raise ValueError("seq_lens must be a contiguous int32 tensor on the cache device")
        if out is None:
            out = torch.empty(self.batch, self.num_q_heads, self.head_dim, dtype=torch.float32, device=self.device)
        if workspace is None:  # (a caller's workspace is sized by the library's own check)
            need = self.workspace_bytes(max_seq_len)
            if self._workspace is None or self._workspace.numel() < need:
                self._workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=self.device)
            workspace = self._workspace
        N.tq_decode_attention(self.desc, q.data_ptr(), seq_lens.data_ptr(), max_seq_len, out.data_ptr(),
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(self.device))
        return out

    def multi_query(self, q: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                    out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
        """Causal attention of the n_query newest tokens of every sequence: fp16 q
        [B, n_query, Hq, d] (query i of sequence b at position seq_lens[b] -
        n_query + i, its K/V already appended); returns float32 [B, n_query, Hq, d]."""
        if (q.dtype != torch.float16 or not q.is_contiguous() or q.dim() != 4 or q.shape[0] != self.batch
                or q.shape[2:] != (self.num_q_heads, self.head_dim)):
            raise ValueError("q must be a contiguous fp16 tensor [B, n_query, Hq, d]")
        if seq_lens.dtype != torch.int32 or seq_lens.device != self.device or not seq_lens.is_contiguous():
            raise ValueError("seq_lens must be a contiguous int32 tensor on the cache device")
        nq = q.shape[1]
        if out is None:
            out = torch.empty(self.batch, nq, self.num_q_heads, self.head_dim, dtype=torch.float32,
                              device=self.device)
        if workspace is None:
            need = N.tq_multi_query_workspace_bytes(self.desc, nq, max_seq_len)
            if self._workspace is None or self._workspace.numel() < need:
                self._workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=self.device)
            workspace = self._workspace
        N.tq_multi_query_attention(self.desc, q.data_ptr(), nq, seq_lens.data_ptr(), max_seq_len, out.data_ptr(),
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   _stream_handle(self.device))
        return out

    # -- inspection -------------------------------------------------------------
    def dequantize(self, which: int, b: int, seq_len: int, token_start: int, n_tokens: int) -> torch.Tensor:
        """float32 [Hkv, n_tokens, d] of positions [token_start, token_start + n_tokens) of sequence b."""
        out = torch.empty(self.num_kv_heads, max(n_tokens, 1), self.head_dim, dtype=torch.float32,
                          device=self.device)
        N.tq_dequantize(self.desc, which, b, seq_len, token_start, n_tokens, out.data_ptr(),
                        _stream_handle(self.device))
        return out[:, :n_tokens]

    def device_status(self) -> int:
        """OR of the TQ_DEV_ERR_* bits raised by the kernels so far (synchronizes)."""
        return int(self.status.item())
