"""One DDTree verification round on the GPU: the five C-ABI calls in stream order.

`Round` owns the device buffers of one synthetic workload (drafter logits, tree-row
projections, prefix caches, GDN inputs and state, target logits), preallocates every
output and workspace once, and `step()` enqueues build -> tree attention -> tree GDN
-> walk -> commit with no host synchronisation.  The synthetic layers are independent,
so each attention/GDN call covers all layers at once (a model would call per layer).

All arithmetic is in libddt.so; this module only allocates and passes pointers.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import ddt, synth


class Round:
    def __init__(self, cfg: dict, device="cuda", workload: int = 5, prefix=None, poison: bool = False,
                 attn_out_dtype=None, gdn_out_dtype=None):
        self.cfg = c = dict(cfg)
        dev = self.device = torch.device(device)
        B, D, V, k, budget = c["B"], c["D"], c["V"], c["top_k"], c["budget"]
        N = self.N = budget + 1
        dt = c["dtype"]
        self.A = D + 1
        if prefix is None:
            if "P" in c:
                prefix = np.full(B, c["P"], np.int32)
            elif "P_lo" in c:
                prefix = synth.prefix_lengths(B, c["P_lo"], c["P_hi"], g=synth.gen(workload, 2)).numpy()
            else:                      # no attention layers: the prefix only sets positions
                prefix = np.zeros(B, np.int32)
        prefix = np.asarray(prefix, np.int32)
        self.prefix0 = torch.as_tensor(prefix).to(dev)
        self.prefix_len = self.prefix0.clone()
        self.Pcap = int(c.get("Pcap", int(prefix.max()) + self.A))
        self.page = int(c.get("page", 0))   # > 0: paged prefix caches of this many rows a page
        if self.page:
            self.Pcap = -(-self.Pcap // self.page) * self.page
        i32 = dict(dtype=torch.int32, device=dev)
        # drafter output and round roots
        self.draft_logits = synth.draft_logits(B, D, V, std=c.get("logit_std", 3.0), boost=c.get("boost", 6.0),
                                               g=synth.gen(workload, 1, dev), dtype=dt, device=dev)
        self.root_token = torch.randint(0, V, (B,), generator=synth.gen(workload, 3, dev), device=dev,
                                        dtype=torch.int32)
        # target logits per tree row
        self.target_logits = synth.target_logits(B, N, V, g=synth.gen(workload, 30, dev), dtype=dt, device=dev)
        # full-attention layers
        self.Lf = c.get("Lf", 0)
        if self.Lf:
            self.attn = synth.attn_inputs(self.Lf, B, N, c["Hq"], c["Hkv"], c["d"], self.Pcap, prefix,
                                          workload=workload, dtype=dt, device=dev, poison=poison)
            self.attn_o = torch.empty((self.Lf, B, N, c["Hq"], c["d"]), dtype=attn_out_dtype or dt, device=dev)
            self.attn_status = torch.empty((B,), **i32)
            ws = ddt.load().ddt_tree_attn_workspace(self.Lf, B, N, c["Hq"], c["Hkv"], c["d"], self.Pcap)
            if c.get("rope"):
                ws = ddt.rope_workspace_bytes(ws, B, N, int(c["rope"]))
            self.attn_ws = torch.empty(max(16, ws), dtype=torch.uint8, device=dev)
            if self.page:
                self._to_pages(workload)
        # GDN layers (state stored [dv][dk])
        self.Lg = c.get("Lg", 0)
        if self.Lg:
            g = synth.gdn_inputs(self.Lg, B, N, c["Hk"], c["Hv"], c["dk"], c["dv"], c["conv_k"], workload=workload,
                                 dtype=dt, device=dev)
            g.S = g.S.transpose(-1, -2).contiguous()
            self.gdn = g
            self.gdn_o = torch.empty((self.Lg, B, N, c["Hv"], c["dv"]), dtype=gdn_out_dtype or dt, device=dev)
            self.gdn_status = torch.empty((B,), **i32)
        # outputs of build / walk / commit
        W = (N + 31) // 32
        self.tree = {"token": torch.empty((B, N), **i32), "parent": torch.empty((B, N), **i32),
                     "depth": torch.empty((B, N), **i32), "position": torch.empty((B, N), **i32),
                     "n_nodes": torch.empty((B,), **i32), "anc": torch.empty((B, N, W), **i32),
                     "score": torch.empty((B, N), dtype=torch.float64, device=dev),
                     "status": torch.empty((B,), **i32)}
        lib = ddt.load()
        self.build_ws = torch.empty(max(16, lib.ddt_build_tree_workspace(B, D, V, k)), dtype=torch.uint8, device=dev)
        self.walk = {"target_argmax": torch.empty((B, N), **i32), "acc_nodes": torch.empty((B, self.A), **i32),
                     "acc_len": torch.empty((B,), **i32), "bonus": torch.empty((B,), **i32),
                     "emitted": torch.empty((B, self.A), **i32), "n_emitted": torch.empty((B,), **i32),
                     "status": torch.empty((B,), **i32)}
        self.temperature = float(c.get("temperature", 0.0))   # > 0: the sampling walk
        if self.temperature > 0:
            self.uniforms = synth.uniforms(B, self.A, k, g=synth.gen(workload, 33, dev), device=dev)
            ws = lib.ddt_walk_accept_sample_workspace(B, N, V)
        else:
            ws = lib.ddt_walk_accept_workspace(B, N, V)
        self.walk_ws = torch.empty(max(16, ws), dtype=torch.uint8, device=dev)
        self.commit = {"src_row": torch.empty((B, self.A), **i32), "dst_pos": torch.empty((B, self.A), **i32),
                       "status": torch.empty((B,), **i32)}

    def _to_pages(self, workload):
        """Move the contiguous caches into head-major pages [L][num_pages][Hkv][page][d]
        behind a shuffled block table (two spare pages), one layer at a time."""
        a, pg = self.attn, self.page
        L, B, Hkv, Pcap, d = a.k_cache.shape
        mp = Pcap // pg
        num = B * mp + 2
        g = synth.gen(workload, 60)
        self.block_table = torch.randperm(num, generator=g)[:B * mp].reshape(B, mp).to(torch.int32).to(self.device)
        phys = self.block_table.flatten().long()
        self.k_pages = torch.empty((L, num, Hkv, pg, d), dtype=a.k_cache.dtype, device=self.device)
        self.v_pages = torch.empty_like(self.k_pages)
        for src, dst in ((a.k_cache, self.k_pages), (a.v_cache, self.v_pages)):
            for l in range(L):
                dst[l, phys] = src[l].reshape(B, Hkv, mp, pg, d).transpose(1, 2).reshape(B * mp, Hkv, pg, d)
        a.k_cache = a.v_cache = None

    # ------------------------------------------------------------------ the round
    def step(self, wait=None):
        """One round.  wait(name), if given, is called before the call that first reads the
        inputs of group `name` ("build", "attn", "gdn", "walk"; see input_groups)."""
        c = self.cfg
        if wait:
            wait("build")
        ddt.ddt_build_tree(self.draft_logits, self.root_token, self.prefix_len, c["top_k"], c["budget"],
                           out=self.tree, workspace=self.build_ws)
        if wait and self.Lf:
            wait("attn")
        self.attention()
        if self.Lg:
            if wait:
                wait("gdn")
            g = self.gdn
            ddt.ddt_tree_gdn(g.x, g.conv_w, g.conv_state, g.beta, g.decay, g.S, self.tree["parent"],
                             self.tree["n_nodes"], Hk=c["Hk"], out_dtype=self.gdn_o.dtype, out=self.gdn_o,
                             status=self.gdn_status)
        if wait:
            wait("walk")
        self.walk_step()
        kw = {}
        if self.Lf and not self.page:
            kw.update(k_tree=self.attn.k_tree, v_tree=self.attn.v_tree, k_cache=self.attn.k_cache,
                      v_cache=self.attn.v_cache)
        if self.Lg:
            g = self.gdn
            kw.update(x=g.x, conv_w=g.conv_w, beta=g.beta, decay=g.decay, S=g.S, conv_state=g.conv_state,
                      Hk=c["Hk"])
        if not (self.Lf or self.Lg):
            return                     # nothing is cached: the round ends with the walk
        if self.Lf and self.page:
            ddt.ddt_commit_paged(self.walk["acc_nodes"], self.walk["acc_len"], self.prefix_len, self.block_table,
                                 k_tree=self.attn.k_tree, v_tree=self.attn.v_tree, k_pages=self.k_pages,
                                 v_pages=self.v_pages, out=self.commit, **kw)
        else:
            ddt.ddt_commit(self.walk["acc_nodes"], self.walk["acc_len"], self.prefix_len, out=self.commit, **kw)

    def walk_step(self):
        """The round's walk: greedy (or its flat safe mode), or rejection sampling at
        cfg["temperature"] with this round's uniforms."""
        t = self.tree
        if self.temperature > 0:
            ddt.ddt_walk_accept_sample(t["token"], t["parent"], t["n_nodes"], self.A - 1,
                                       target_logits=self.target_logits, uniforms=self.uniforms,
                                       temperature=self.temperature, out=self.walk, workspace=self.walk_ws)
        else:
            ddt.ddt_walk_accept(t["token"], t["parent"], t["n_nodes"], self.A - 1, target_logits=self.target_logits,
                                out=self.walk, workspace=self.walk_ws, flat=bool(self.cfg.get("flat", False)))

    def attention(self):
        """The round's attention call.  With cfg["rope"] (rotated channels) q and the tree
        keys are taken before rotary embedding: the keys are rotated in place at their
        positions (they are committed), and q inside the fused attention call."""
        if not self.Lf:
            return
        c, a = self.cfg, self.attn
        scale = 1.0 / math.sqrt(c["d"])
        rot = int(c.get("rope", 0))
        if rot:
            ddt.ddt_rope_tree(None, a.k_tree, self.tree["position"], self.tree["n_nodes"], rot_dim=rot, Hq=c["Hq"])
        common = dict(scale=scale, out_dtype=self.attn_o.dtype, out=self.attn_o, status=self.attn_status,
                      workspace=self.attn_ws)
        if self.page and rot:
            ddt.ddt_tree_attn_paged_rope(a.q, a.k_tree, a.v_tree, self.k_pages, self.v_pages, self.block_table,
                                         self.prefix_len, self.tree["n_nodes"], self.tree["anc"], self.tree["position"],
                                         rot_dim=rot, **common)
        elif self.page:
            ddt.ddt_tree_attn_paged(a.q, a.k_tree, a.v_tree, self.k_pages, self.v_pages, self.block_table,
                                    self.prefix_len, self.tree["n_nodes"], self.tree["anc"], **common)
        elif rot:
            ddt.ddt_tree_attn_rope(a.q, a.k_tree, a.v_tree, a.k_cache, a.v_cache, self.prefix_len, self.tree["n_nodes"],
                                   self.tree["anc"], self.tree["position"], rot_dim=rot, **common)
        else:
            ddt.ddt_tree_attn(a.q, a.k_tree, a.v_tree, a.k_cache, a.v_cache, self.prefix_len, self.tree["n_nodes"],
                              self.tree["anc"], **common)

    def restore_prefix(self):
        """Reset the committed prefix lengths (the commit advanced them)."""
        self.prefix_len.copy_(self.prefix0, non_blocking=True)

    def drafted_nodes(self) -> int:
        return int((self.tree["n_nodes"] - 1).sum())

    # ------------------------------------------------------------ per-round inputs
    def round_inputs(self):
        """The tensors a serving loop hands to each round (everything except the
        persistent caches, GDN state and conv state)."""
        ins = {"draft_logits": self.draft_logits, "root_token": self.root_token, "target_logits": self.target_logits}
        if self.temperature > 0:
            ins["uniforms"] = self.uniforms
        if self.Lf:
            ins.update(q=self.attn.q, k_tree=self.attn.k_tree, v_tree=self.attn.v_tree)
        if self.Lg:
            ins.update(x=self.gdn.x, beta=self.gdn.beta, decay=self.gdn.decay)
        return ins

    def input_groups(self):
        """Names of round_inputs() by the call that first reads them, in call order."""
        g = {"build": ["draft_logits", "root_token"]}
        if self.Lf:
            g["attn"] = ["q", "k_tree", "v_tree"]
        if self.Lg:
            g["gdn"] = ["x", "beta", "decay"]
        g["walk"] = ["target_logits"] + (["uniforms"] if self.temperature > 0 else [])
        return g

    def bind_inputs(self, ins: dict):
        """Point the round at another set of per-round input tensors (same keys, shapes and
        dtypes as `round_inputs()`), e.g. the other half of a double buffer."""
        self.draft_logits, self.root_token, self.target_logits = ins["draft_logits"], ins["root_token"], \
            ins["target_logits"]
        if self.Lf:
            self.attn.q, self.attn.k_tree, self.attn.v_tree = ins["q"], ins["k_tree"], ins["v_tree"]
        if self.Lg:
            self.gdn.x, self.gdn.beta, self.gdn.decay = ins["x"], ins["beta"], ins["decay"]
        if self.temperature > 0:
            self.uniforms = ins["uniforms"]

    def round_outputs(self):
        return {"emitted": self.walk["emitted"], "n_emitted": self.walk["n_emitted"]}
