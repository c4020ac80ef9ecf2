"""Device-side setup of a synthetic workload for the tests, smoke() and the bench.

Takes a dcp_workloads.Workload (host arrays) and builds what a serving engine
would hold on the GPU: the query batch, per-rank block tables over one
physical pool, and the paged cache, filled through libdcp's own slot mapping
and cache write.  torch only allocates and copies; every computation is a
libdcp call.
"""

import numpy as np
import torch

from dcp_workloads import allocate_blocks

from . import (
    dcp_decode_attention, dcp_decode_attention_planned, dcp_decode_plan, dcp_get_error, dcp_lse_merge, dcp_partial_attention, dcp_pcp_partition,
    dcp_prefill_attention, dcp_slot_mapping, dcp_workspace_init, dcp_workspace_size, params_from_config,
)

_TORCH_STORAGE = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}


def raw_to_torch(arr, dtype):
    """Host raw storage (float32 / uint16 bf16 bits / uint8 fp8 bits) as a torch tensor."""
    arr = np.ascontiguousarray(arr)
    if dtype == "bf16":
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(arr)


class DeviceWorkload:
    """A workload resident in HBM: q, paged KV pool, block tables, metadata."""

    def __init__(self, wl, device="cuda:0", populate=True, spare_blocks=0, stream=None, workspace_bytes=None):
        self.wl = wl
        self.cfg = c = wl.cfg
        self.dev = torch.device(device)
        self.stream = stream or torch.cuda.current_stream(self.dev)
        self.params = params_from_config(c, wl.kv_scale)
        self.B, self.Tq, self.Hq = int(c["B"]), int(c["Tq"]), int(c["Hq"])
        self.Hkv, self.Dk, self.Dv = int(c["Hkv"]), int(c["Dk"]), int(c["Dv"])
        self.N, self.bs = int(c["N"]), int(c["block_size"])
        self.mla = c["layout"] == "mla"
        dev = self.dev
        self.seq_lens = torch.from_numpy(wl.seq_lens.astype(np.int32)).to(dev)
        # (prefill needs only the error word; the decode scratch grows with Tq)
        self.ws_bytes = workspace_bytes or dcp_workspace_size(self.params, self.B, int(wl.seq_lens.max()))
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        dcp_workspace_init(self.workspace, self.stream)

        # 1. per-rank lengths and block needs (libdcp metadata)
        self.local_lens = torch.empty((self.N, self.B), dtype=torch.int32, device=dev)
        self.virt_blocks = torch.empty(self.B, dtype=torch.int32, device=dev)
        self.rank_blocks = torch.empty((self.N, self.B), dtype=torch.int32, device=dev)
        dcp_slot_mapping(self.params, self.seq_lens, local_lens=self.local_lens, virt_blocks=self.virt_blocks,
                         rank_blocks=self.rank_blocks, workspace=self.workspace, stream=self.stream)
        self.stream.synchronize()
        # 2. physical blocks: a seeded random permutation of the pool
        tables, self.num_blocks = allocate_blocks(self.rank_blocks.cpu().numpy(), seed=wl.seed,
                                                  spare=spare_blocks)
        self.block_tables_host = tables
        self.block_tables = torch.from_numpy(tables).to(dev)
        # 3. the pool and the query batch
        kvt = _TORCH_STORAGE[c["kv_dtype"]]
        if self.mla:
            self.k_pool = torch.zeros((self.num_blocks, self.bs, self.Dk), dtype=kvt, device=dev)
            self.v_pool = None
        else:
            self.k_pool = torch.zeros((self.num_blocks, self.Hkv, self.bs, self.Dk), dtype=kvt, device=dev)
            self.v_pool = torch.zeros((self.num_blocks, self.Hkv, self.bs, self.Dv), dtype=kvt, device=dev)
        self.q = raw_to_torch(wl.q, c["q_dtype"]).to(dev)
        ot = torch.float32 if c["out_dtype"] == "f32" else torch.bfloat16
        self.out = torch.empty((self.B, self.Tq, self.Hq, self.Dv), dtype=ot, device=dev)
        self.lse = torch.empty((self.B, self.Tq, self.Hq), dtype=torch.float32, device=dev)
        self.out_partial = None
        self.lse_partial = None
        # the newest Tq tokens of every request: the decode step's cache writes
        nr, npos = wl.new_token_lists()
        self.new_req = torch.from_numpy(nr).to(dev)
        self.new_pos = torch.from_numpy(npos).to(dev)
        rows = (wl.req_start[:-1][nr] + npos).astype(np.int64)
        self.new_k = raw_to_torch(wl.k[rows], c["kv_dtype"]).to(dev)
        self.new_v = None if wl.v is None else raw_to_torch(wl.v[rows], c["kv_dtype"]).to(dev)
        if populate:
            self.populate()

    # -- cache fill -------------------------------------------------------------
    def populate(self, chunk_tokens=1 << 20):
        """Write every token of every request into its owner's slot (libdcp scatter)."""
        wl, c = self.wl, self.cfg
        tok_req, tok_pos = wl.token_lists()
        T = tok_req.size
        for s in range(0, T, chunk_tokens):
            e = min(T, s + chunk_tokens)
            req = torch.from_numpy(tok_req[s:e]).to(self.dev)
            pos = torch.from_numpy(tok_pos[s:e]).to(self.dev)
            nk = raw_to_torch(wl.k[s:e], c["kv_dtype"]).to(self.dev)
            nv = None if wl.v is None else raw_to_torch(wl.v[s:e], c["kv_dtype"]).to(self.dev)
            dcp_slot_mapping(self.params, self.seq_lens, req, pos, self.block_tables, self.num_blocks,
                             new_k=nk, new_v=nv, k_pool=self.k_pool, v_pool=self.v_pool,
                             workspace=self.workspace, stream=self.stream)
        self.stream.synchronize()

    # -- the hot path -------------------------------------------------------------
    def write_new_tokens(self):
        """Slot mapping + cache write of the step's Tq new tokens per request."""
        dcp_slot_mapping(self.params, self.seq_lens, self.new_req, self.new_pos, self.block_tables,
                         self.num_blocks, new_k=self.new_k, new_v=self.new_v, k_pool=self.k_pool,
                         v_pool=self.v_pool, workspace=self.workspace, stream=self.stream)

    def decode(self):
        dcp_decode_attention(self.params, self.q, self.k_pool, self.v_pool, self.num_blocks, self.block_tables,
                             self.seq_lens, self.local_lens, self.out, self.lse, self.workspace, self.stream)
        return self.out, self.lse

    def plan_and_write(self):
        """The step's work plan on a second stream while this one writes the new
        tokens (the plan needs the lengths only); this stream waits for both."""
        if getattr(self, "_pstream", None) is None:
            self._pstream = torch.cuda.Stream(device=self.dev)
            self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()
        self._fork.record(self.stream)
        self._pstream.wait_event(self._fork)
        dcp_decode_plan(self.params, self.seq_lens, self.local_lens, int(self.block_tables.shape[-1]),
                        self.workspace, self._pstream)
        self._join.record(self._pstream)
        self.write_new_tokens()
        self.stream.wait_event(self._join)

    def decode_planned(self):
        """Fused attention + merge on the plan plan_and_write made."""
        dcp_decode_attention_planned(self.params, self.q, self.k_pool, self.v_pool, self.num_blocks,
                                     self.block_tables, self.seq_lens, self.local_lens, self.out, self.lse,
                                     self.workspace, self.stream)
        return self.out, self.lse

    def step(self):
        """One decode step: the plan beside the cache write of the new tokens, then
        fused attention + merge."""
        self.plan_and_write()
        return self.decode_planned()

    def partial(self):
        if self.out_partial is None:
            self.out_partial = torch.empty((self.N, self.B, self.Tq, self.Hq, self.Dv), dtype=torch.float32,
                                           device=self.dev)
            self.lse_partial = torch.empty((self.N, self.B, self.Tq, self.Hq), dtype=torch.float32,
                                           device=self.dev)
        dcp_partial_attention(self.params, self.q, self.k_pool, self.v_pool, self.num_blocks, self.block_tables,
                              self.seq_lens, self.local_lens, self.out_partial, self.lse_partial,
                              self.workspace, self.stream)
        return self.out_partial, self.lse_partial

    def merge(self, out=None, lse=None):
        """dcp_lse_merge of the current partials into out/lse."""
        rows = self.B * self.Tq * self.Hq
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        dcp_lse_merge(self.N, rows, self.Dv, self.out_partial, self.lse_partial, out, self.params.out_dtype, lse,
                      self.stream)
        return out, lse

    # -- prefill of the newest Tq tokens under PCP (head-tail partition) ---------
    def prefill_setup(self, K):
        """The chunk = every request's newest Tq tokens.  Runs the partition
        over K PCP ranks once and lays the query rows out in the gathered
        order (what an AllGather of the ranks' queries produces): an input
        permutation, done once."""
        B, Tq = self.B, self.Tq
        self.pcp_K = int(K)
        self.max_q = -(-Tq // (2 * self.pcp_K)) * 2 * self.pcp_K
        self.ctx_lens = (self.seq_lens - Tq).to(torch.int32)
        self.q_lens = torch.full((B,), Tq, dtype=torch.int32, device=self.dev)
        self.q_pos = torch.empty((B, self.max_q), dtype=torch.int32, device=self.dev)
        self.padded_lens = torch.empty(B, dtype=torch.int32, device=self.dev)
        self.partition()
        pos = self.q_pos.long()
        natural = (pos - self.ctx_lens.long()[:, None]).clamp(min=0)
        qg = torch.gather(self.q, 1, natural[:, :, None, None].expand(B, self.max_q, self.Hq, self.Dk))
        self.q_gathered = torch.where((pos >= 0)[:, :, None, None], qg, torch.zeros_like(qg)).contiguous()
        self.p_out = torch.empty((self.N, B, self.max_q, self.Hq, self.Dv), dtype=torch.float32, device=self.dev)
        self.p_lse = torch.empty((self.N, B, self.max_q, self.Hq), dtype=torch.float32, device=self.dev)
        ot = torch.float32 if self.cfg["out_dtype"] == "f32" else torch.bfloat16
        self.g_out = torch.empty((B, self.max_q, self.Hq, self.Dv), dtype=ot, device=self.dev)
        self.g_lse = torch.empty((B, self.max_q, self.Hq), dtype=torch.float32, device=self.dev)

    def partition(self):
        dcp_pcp_partition(self.pcp_K, self.ctx_lens, self.q_lens, self.max_q, self.q_pos, self.padded_lens,
                          workspace=self.workspace, stream=self.stream)

    def prefill(self, merged=True):
        """One prefill attention pass: partition, per-rank causal partials, merge."""
        self.partition()
        dcp_prefill_attention(self.params, self.q_gathered, self.q_pos, self.k_pool, self.v_pool, self.num_blocks,
                              self.block_tables, self.seq_lens, self.local_lens, self.p_out, self.p_lse,
                              self.g_out if merged else None, self.g_lse if merged else None,
                              workspace=self.workspace, stream=self.stream)
        return self.g_out, self.g_lse

    def slot_mapping(self, tok_req, tok_pos):
        """owner / slots for given tokens (host arrays in, device tensors out)."""
        T = len(tok_req)
        req = torch.from_numpy(np.ascontiguousarray(tok_req, dtype=np.int32)).to(self.dev)
        pos = torch.from_numpy(np.ascontiguousarray(tok_pos, dtype=np.int64)).to(self.dev)
        owner = torch.empty(T, dtype=torch.int8, device=self.dev)
        slots = torch.empty((self.N, T), dtype=torch.int64, device=self.dev)
        dcp_slot_mapping(self.params, self.seq_lens, req, pos, self.block_tables, self.num_blocks, owner=owner,
                         slots=slots, workspace=self.workspace, stream=self.stream)
        return owner, slots

    def error_bits(self):
        return dcp_get_error(self.workspace, self.stream)
