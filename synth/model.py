"""The synthetic stand-in for a language model: it knows every request's token
sequence (prompt, then the tokens it generates) and supplies the Q/K/V rows of
any positions, computed from prefix hashes.  Values come from the GPU kernel
of synth/csrc/synth_gen.cu (the same definition as synth/hashgen.py).
"""
from __future__ import annotations

import numpy as np

from . import native
from .hashgen import KIND_K, KIND_Q, KIND_V, root_hash


class SynthModel:
    def __init__(self, shape, seed: int, vocab: int, device="cuda"):
        import torch
        self.torch = torch
        self.shape = shape
        self.seed = seed
        self.vocab = vocab
        self.h0 = root_hash(seed)
        self.device = torch.device(device)
        self._hashes = {}

    # ---------------------------------------------------------------- host
    def sequence(self, prompt: np.ndarray, max_new: int):
        """Prompt followed by the max_new tokens the model generates; and the
        prefix hash of every position."""
        prompt = np.ascontiguousarray(prompt, np.int32)
        h = native.prefix_hashes_from(self.h0, prompt)
        if max_new:
            toks, hs = native.decode_tokens(int(h[-1]) if len(h) else self.h0, max_new, self.vocab)
            return np.concatenate([prompt, toks]).astype(np.int32), np.concatenate([h, hs])
        return prompt, h

    def register(self, rid: int, hashes: np.ndarray):
        self._hashes[rid] = hashes

    def hashes(self, rid: int) -> np.ndarray:
        return self._hashes[rid]

    # -------------------------------------------------------------- device
    def rows(self, hashes: np.ndarray, kinds=("q", "k", "v")):
        """Device Q/K/V rows for the given position hashes."""
        torch = self.torch
        sh = self.shape
        n = len(hashes)
        dh = torch.from_numpy(np.ascontiguousarray(hashes).view(np.int64)).to(self.device)
        out = {}
        if "q" in kinds:
            q = torch.empty(n, sh.q_heads, sh.head_dim_k, dtype=torch.bfloat16, device=self.device)
            native.gen_values_gpu(dh, KIND_Q, sh.q_heads, sh.head_dim_k, q.view(n, -1))
            out["q"] = q
        if "k" in kinds:
            if sh.mla:
                k = torch.empty(n, sh.head_dim_k, dtype=torch.bfloat16, device=self.device)
                native.gen_values_gpu(dh, KIND_K, 1, sh.head_dim_k, k)
            else:
                k = torch.empty(n, sh.kv_heads, sh.head_dim_k, dtype=torch.bfloat16, device=self.device)
                native.gen_values_gpu(dh, KIND_K, sh.kv_heads, sh.head_dim_k, k.view(n, -1))
            out["k"] = k
        if "v" in kinds:
            if sh.mla:
                out["v"] = None
            else:
                v = torch.empty(n, sh.kv_heads, sh.head_dim_v, dtype=torch.bfloat16, device=self.device)
                native.gen_values_gpu(dh, KIND_V, sh.kv_heads, sh.head_dim_v, v.view(n, -1))
                out["v"] = v
        return out

    def extend_inputs(self, batch):
        hs = [self._hashes[r.rid][r.first:r.prompt_len] for r in batch]
        h = np.concatenate(hs) if hs else np.zeros(0, np.uint64)
        return self.rows(h)

    def extend_kv(self, batch):
        """K/V rows only (a prefill that stores K/V without attention)."""
        hs = [self._hashes[r.rid][r.first:r.prompt_len] for r in batch]
        h = np.concatenate(hs) if hs else np.zeros(0, np.uint64)
        return self.rows(h, kinds=("k", "v"))

    def decode_inputs(self, batch, t: int):
        h = np.asarray([self._hashes[r.rid][r.prompt_len + t] for r in batch], np.uint64)
        return self.rows(h)

    def kv_rows(self, hashes):
        return self.rows(hashes, kinds=("k", "v"))
