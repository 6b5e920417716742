"""A module-style holder of the selector's weights, named as on the source page.

Page "vllm.models.beam.nvidia.dflash2", class DFlash2BeamCandidateSelector: it owns the
predecessor and successor codebooks ([vocab, rank]) and the bias-free hidden projection
(hidden_size -> rank, weight [rank, hidden_size]), all bf16, and forward(candidate_ids,
unary_logits, hidden_states, anchor_token_ids) returns the edge scores [requests, steps, top_k
(predecessor), top_k]. This class keeps the same names and shapes and runs every step through
the library's C ABI; it holds tensors and marshals arguments, nothing more.
"""

from __future__ import annotations

import torch

from . import (dflash_best_path, dflash_lmhead_topk, dflash_selector, dflash_selector_forward,
               dflash_selector_lmhead)


class CandidateSelector:
    """Weights of the low-rank candidate selector on one CUDA device.

    predecessor_codebook, successor_codebook: [vocab_size, rank] bf16.
    hidden_projection_weight: [rank, hidden_size] bf16 (a Linear's [out, in] weight).
    The tensors are allocated uninitialised; load or assign the weights before use.
    """

    def __init__(self, hidden_size: int, vocab_size: int, rank: int, top_k: int,
                 device: torch.device | str | None = None,
                 params_dtype: torch.dtype = torch.bfloat16):
        if params_dtype != torch.bfloat16:
            raise NotImplementedError("the selector's weights are bf16")
        dev = torch.device(device) if device is not None else torch.device("cuda")
        self.hidden_size = hidden_size
        self.vocab_size = vocab_size
        self.rank = rank
        self.top_k = top_k
        self.predecessor_codebook = torch.empty((vocab_size, rank), dtype=params_dtype, device=dev)
        self.successor_codebook = torch.empty((vocab_size, rank), dtype=params_dtype, device=dev)
        self.hidden_projection_weight = torch.empty((rank, hidden_size), dtype=params_dtype,
                                                    device=dev)

    def forward(self, candidate_ids: torch.Tensor, unary_logits: torch.Tensor,
                hidden_states: torch.Tensor, anchor_token_ids: torch.Tensor) -> torch.Tensor:
        """Edge scores [R, S, top_k, top_k] of given candidates (dflash_selector_forward)."""
        if hidden_states.dtype != torch.bfloat16:
            raise ValueError("hidden_states must be bf16")
        _, edges = dflash_selector_forward(candidate_ids, unary_logits, hidden_states,
                                           anchor_token_ids, self.hidden_projection_weight,
                                           self.predecessor_codebook, self.successor_codebook)
        return edges

    __call__ = forward

    def select(self, logits: torch.Tensor, hidden_states: torch.Tensor,
               anchor_token_ids: torch.Tensor, softcap: float = 0.0, scale: float = 1.0):
        """Candidates from logits [R, S, V] and their edge scores in one call
        (dflash_selector): returns (candidate_ids, unary_logits, edges)."""
        ids, unary, _, edges = dflash_selector(
            logits, hidden_states, self.hidden_projection_weight, self.predecessor_codebook,
            self.successor_codebook, anchor_token_ids, self.top_k, softcap=softcap, scale=scale)
        return ids, unary, edges

    def compute_candidates(self, hidden_states: torch.Tensor, lm_head: torch.Tensor,
                           softcap: float = 0.0, scale: float = 1.0):
        """The top_k candidate ids and their (processed) logits at each position, straight
        from the LM head [V, H] without logits in memory, as the page's
        DFlash2BeamForCausalLM.compute_candidates gives them (dflash_lmhead_topk)."""
        return dflash_lmhead_topk(hidden_states, lm_head, self.top_k, softcap=softcap,
                                  scale=scale)

    def select_from_lm_head(self, hidden_states: torch.Tensor, lm_head: torch.Tensor,
                            anchor_token_ids: torch.Tensor, softcap: float = 0.0,
                            scale: float = 1.0):
        """Candidates straight from the LM head [V, H] (no logits in memory) and their edge
        scores in one call (dflash_selector_lmhead): returns (candidate_ids, unary_logits,
        edges)."""
        ids, unary, _, edges = dflash_selector_lmhead(
            hidden_states, lm_head, self.hidden_projection_weight, self.predecessor_codebook,
            self.successor_codebook, anchor_token_ids, self.top_k, softcap=softcap, scale=scale)
        return ids, unary, edges

    @staticmethod
    def best_path(edges: torch.Tensor, candidate_ids: torch.Tensor):
        """The max-sum path through the edge scores (dflash_best_path): returns (path, tokens,
        score)."""
        return dflash_best_path(edges, candidate_ids)
