"""Device-memory plumbing around the C ABI: torch allocates the caller-owned buffers
(weights, workspace, paged KV, boundary, outputs) and every call goes through
``binding`` into libeagle3.so.  No arithmetic of the method happens here."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .synth import DrafterWeights, Geometry


def _dev_bits(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream


class DraftModel:
    """Drafter weights resident in HBM plus one library context."""

    KV_FORMATS = {"bf16": B.EAGLE3_KV_BF16, "q8_0/q5_1": B.EAGLE3_KV_Q8_0_Q5_1}

    def __init__(self, weights: DrafterWeights, max_batch: int, max_gamma: int,
                 max_cache_len: int, page_size: int, device="cuda", stream=None,
                 kv_format: str = "bf16", flags: int = 0):
        if not torch.cuda.is_available():
            raise RuntimeError("DraftModel needs a CUDA device")
        self.geom: Geometry = weights.geom
        self.device = torch.device(device)
        g = self.geom
        self.cfg = B.Config(n_embd=g.n_embd, n_head=g.n_head, n_head_kv=g.n_head_kv,
                            head_dim=g.head_dim, rope_dims=g.rope_dims,
                            rope_theta=g.rope_theta, rms_eps=g.rms_eps, n_ff=g.n_ff,
                            draft_vocab=g.draft_vocab, target_vocab=g.target_vocab,
                            max_batch=max_batch, max_gamma=max_gamma,
                            max_cache_len=max_cache_len, page_size=page_size,
                            flags=flags, kv_format=self.KV_FORMATS[kv_format],
                            weight_format=B.EAGLE3_W_INT4_G128 if weights.int4 else B.EAGLE3_W_BF16)
        self.kv_format = kv_format
        self.max_batch, self.max_gamma = max_batch, max_gamma
        self.max_cache_len, self.page_size = max_cache_len, page_size
        self.w = {name: _dev_bits(b, self.device) for name, b in weights.bits.items()}
        self.w_sz = {}
        for name, (codes, sz) in (weights.int4 or {}).items():  # INT4 projections
            self.w[name] = torch.from_numpy(np.ascontiguousarray(codes)).to(self.device)
            self.w_sz[name] = torch.from_numpy(np.ascontiguousarray(sz).view(np.int32)).to(self.device)
        self.d2t = torch.from_numpy(np.ascontiguousarray(weights.d2t)).to(self.device)
        ws_bytes = B.eagle3_workspace_bytes(self.cfg)
        if ws_bytes == 0:
            raise B.Eagle3Error(B.EAGLE3_ERR_UNSUPPORTED, "eagle3_workspace_bytes")
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        wt = B.Weights(**{f: self.w[f].data_ptr() for f in B.WEIGHT_FIELDS if f != "d2t"},
                       d2t=self.d2t.data_ptr(),
                       **{f"{k}_sz": v.data_ptr() for k, v in self.w_sz.items()})
        self._weights_struct = wt
        self.ctx = B.eagle3_init(self.cfg, wt, self.workspace.data_ptr(), ws_bytes,
                                 _stream_handle(stream))

    def close(self):
        if getattr(self, "ctx", None):
            B.eagle3_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- state objects
    def new_state(self, batch: int, page_table: np.ndarray | None = None,
                  num_pages: int | None = None) -> "SeqBatch":
        return SeqBatch(self, batch, page_table, num_pages)

    # ---------------------------------------------------------------- entry points
    def encode(self, aux: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        M = aux.shape[0]
        if out is None:
            out = torch.empty(M, self.geom.n_embd, dtype=torch.float32, device=self.device)
        B.eagle3_encode(self.ctx, aux.data_ptr(), M, out.data_ptr(), _stream_handle(stream))
        return out

    def set_graph_mode(self, on: bool):
        B.eagle3_set_graph_mode(self.ctx, on)

    def set_tc_min_items(self, min_items: int):
        """Items from which projections use the tensor cores (0: the default)."""
        B.eagle3_set_tc_min_items(self.ctx, min_items)

    def set_attention(self, mode: int):
        """Decode attention kernel for a bf16 KV cache: 0 CUDA cores (the default),
        1 tensor cores where they apply."""
        B.eagle3_set_attention(self.ctx, mode)

    def set_tc_schedule(self, schedule: int):
        """Tile schedule of the tensor-core projections: 0 automatic, 1 stream-K,
        2 cluster split-K wherever it fits."""
        B.eagle3_set_tc_schedule(self.ctx, schedule)

    def status(self) -> int:
        return B.eagle3_get_status(self.ctx)


class SeqBatch:
    """Paged KV cache, committed lengths and boundary of B sequences, plus the host
    mirror of kv_len that the capacity check reads."""

    def __init__(self, model: DraftModel, batch: int, page_table=None, num_pages=None):
        g, dev = model.geom, model.device
        self.model, self.B = model, batch
        ps = model.page_size
        pages_per_seq = (model.max_cache_len + ps - 1) // ps
        if page_table is None:
            page_table = np.arange(batch * pages_per_seq, dtype=np.int32).reshape(batch, pages_per_seq)
        page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        self.num_pages = int(num_pages if num_pages is not None else page_table.max() + 1)
        self.page_table_host = page_table
        self.page_table = torch.from_numpy(page_table).to(dev)
        k_row, v_row = B.eagle3_kv_row_bytes(model.cfg)
        self.k_pool = torch.zeros(self.num_pages, g.n_head_kv, ps, k_row, dtype=torch.uint8, device=dev)
        self.v_pool = torch.zeros(self.num_pages, g.n_head_kv, ps, v_row, dtype=torch.uint8, device=dev)
        self.kv_len = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.kv_len_host = np.zeros(batch, dtype=np.int32)
        self.g = torch.zeros(batch, g.n_embd, dtype=torch.float32, device=dev)
        self.tok = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.kv = B.KV(k_pool=self.k_pool.data_ptr(), v_pool=self.v_pool.data_ptr(),
                       page_table=self.page_table.data_ptr(), num_pages=self.num_pages,
                       max_pages_per_seq=page_table.shape[1], kv_len=self.kv_len.data_ptr())
        self.bnd = B.Boundary(g=self.g.data_ptr(), tok=self.tok.data_ptr())

    def prefill(self, tokens: torch.Tensor, next_tok: torch.Tensor, prompt_len, aux: torch.Tensor,
                stream=None):
        pl = np.asarray(prompt_len, dtype=np.int32)
        B.eagle3_prefill(self.model.ctx, self.B, tokens.data_ptr(), tokens.shape[1],
                         next_tok.data_ptr(), pl, aux.data_ptr(), self.kv, self.bnd,
                         _stream_handle(stream))
        self.kv_len_host = pl - 1

    def draft_chain(self, gamma: int, flags: int = 0, out: dict | None = None, debug=False,
                    stream=None) -> dict:
        m, dev = self.model, self.model.device
        if out is None:
            out = {"draft_tok": torch.empty(self.B, gamma, dtype=torch.int32, device=dev),
                   "draft_id": torch.empty(self.B, gamma, dtype=torch.int32, device=dev),
                   "gamma_eff": torch.empty(self.B, dtype=torch.int32, device=dev)}
            if debug:
                out["logits"] = torch.empty(self.B, gamma, m.geom.draft_vocab, dtype=torch.float32, device=dev)
                out["g"] = torch.empty(self.B, gamma, m.geom.n_embd, dtype=torch.float32, device=dev)
        ptr = lambda k: out[k].data_ptr() if k in out else None
        B.eagle3_draft_chain(m.ctx, self.B, gamma, flags, self.kv_len_host, self.kv, self.bnd,
                             out["draft_tok"].data_ptr(), ptr("draft_id"), ptr("gamma_eff"),
                             ptr("logits"), ptr("g"), _stream_handle(stream))
        self._gamma_eff_host = np.array([B.eagle3_plan_gamma(int(l), gamma, m.max_cache_len, flags)
                                         for l in self.kv_len_host], dtype=np.int32)
        self._round_start_host = self.kv_len_host.copy()
        self.kv_len_host = self.kv_len_host + self._gamma_eff_host
        return out

    def rewind(self, stream=None):
        B.eagle3_rewind(self.model.ctx, self.B, self.kv, _stream_handle(stream))
        self.kv_len_host = self._round_start_host.copy()

    def accept(self, draft_tok, target_pred, gamma_eff=None, n_acc=None, bonus=None, stream=None):
        dev = self.model.device
        gamma = draft_tok.shape[1]
        n_acc = n_acc if n_acc is not None else torch.empty(self.B, dtype=torch.int32, device=dev)
        bonus = bonus if bonus is not None else torch.empty(self.B, dtype=torch.int32, device=dev)
        B.eagle3_accept(self.model.ctx, self.B, gamma, draft_tok.data_ptr(), target_pred.data_ptr(),
                        gamma_eff.data_ptr() if gamma_eff is not None else None,
                        n_acc.data_ptr(), bonus.data_ptr(), _stream_handle(stream))
        return n_acc, bonus

    def verify_greedy(self, target_lm_head, target_norm, hidden, draft_tok, gamma_eff=None,
                      target_rms_eps=None, target_pred=None, n_acc=None, bonus=None,
                      logits=False, stream=None):
        """Target-side greedy verify of the drafted window: target_pred [B, gamma + 1] (the
        target head's argmax at each window position of `hidden` [B, gamma + 1, n] float32),
        then the accept walk.  target_lm_head / target_norm: bf16 bits as int16 tensors."""
        dev = self.model.device
        gamma = draft_tok.shape[1]
        eps = self.model.geom.rms_eps if target_rms_eps is None else target_rms_eps
        V = int(target_lm_head.shape[0])
        target_pred = target_pred if target_pred is not None else \
            torch.empty(self.B, gamma + 1, dtype=torch.int32, device=dev)
        n_acc = n_acc if n_acc is not None else torch.empty(self.B, dtype=torch.int32, device=dev)
        bonus = bonus if bonus is not None else torch.empty(self.B, dtype=torch.int32, device=dev)
        lg = torch.empty(self.B, gamma + 1, V, dtype=torch.float32, device=dev) if logits else None
        B.eagle3_verify_greedy(self.model.ctx, self.B, gamma, target_lm_head.data_ptr(),
                               target_norm.data_ptr(), eps, hidden.data_ptr(), draft_tok.data_ptr(),
                               gamma_eff.data_ptr() if gamma_eff is not None else None,
                               target_pred.data_ptr(), n_acc.data_ptr(), bonus.data_ptr(),
                               lg.data_ptr() if lg is not None else None, _stream_handle(stream))
        return target_pred, n_acc, bonus, lg

    def rebuild_after_verify(self, n_acc, draft_tok, bonus, verify_aux, n_acc_host=None,
                             stream=None):
        gamma = draft_tok.shape[1]
        B.eagle3_rebuild_after_verify(self.model.ctx, self.B, gamma, n_acc.data_ptr(),
                                      draft_tok.data_ptr(), bonus.data_ptr(),
                                      verify_aux.data_ptr(), self.kv, self.bnd,
                                      _stream_handle(stream))
        if n_acc_host is None:
            n_acc_host = n_acc.cpu().numpy()  # the caller's scheduler knows this; tests sync
        self.kv_len_host = self.kv_len_host + np.asarray(n_acc_host, dtype=np.int32) + 1

    # ---------------------------------------------------------------- inspection
    def kv_entries(self, b: int, lo: int, hi: int):
        """Stored K and V rows of sequence b at positions lo..hi-1: bf16 bits
        [hi - lo, H_kv, d] (uint16), or the q8_0 / q5_1 row bytes [hi - lo, H_kv, row]."""
        return self.kv_entries_at(b, np.arange(lo, hi))

    def kv_entries_at(self, b: int, positions):
        """Stored K and V rows of sequence b at the given positions (any order), in the
        layout of kv_entries."""
        ps = self.model.page_size
        pos = np.asarray(positions, dtype=np.int64)
        pages = torch.from_numpy(self.page_table_host[b, pos // ps].astype(np.int64)).to(self.k_pool.device)
        slots = torch.from_numpy((pos % ps).astype(np.int64)).to(self.k_pool.device)
        k = self.k_pool[pages, :, slots, :].cpu().numpy()
        v = self.v_pool[pages, :, slots, :].cpu().numpy()
        if self.model.kv_format == "bf16":
            return k.view(np.uint16), v.view(np.uint16)
        return k, v
