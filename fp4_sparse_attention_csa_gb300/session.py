"""Device-side state for one workload: torch-allocated pools, page table,
FP8 window, pending tokens and workspaces, filled through csa_append and read
through csa_decode.  Plumbing only: every computation is a libcsa call."""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from . import (KV_PAGE_BYTES, IDX_PAGE_BYTES, OP_APPEND, OP_DECODE, csa_append, csa_append_compress,
               make_compress, csa_decode, csa_step, csa_step_ex,
               csa_workspace_size, make_cache, make_rows, make_window)


def _dev(a, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def _bits_to_bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits)).to(device).view(torch.bfloat16)


class DeviceState:
    def __init__(self, wl, device="cuda", window=True):
        self.wl = wl
        self.device = device
        self.kv_pool = torch.zeros(wl.num_pages * KV_PAGE_BYTES, dtype=torch.uint8, device=device)
        self.idx_pool = torch.zeros(wl.num_pages * IDX_PAGE_BYTES, dtype=torch.uint8, device=device)
        self.page_table = _dev(wl.page_table, torch.int32, device)
        self.cache = make_cache(self.kv_pool, self.idx_pool, self.page_table, wl.num_pages, wl.P)
        self.win_codes = self.win_scale = None
        self.window = None
        if window:
            self.win_codes = torch.zeros(wl.B * wl.win_cap * 512, dtype=torch.uint8, device=device)
            self.win_scale = torch.zeros(wl.B * wl.win_cap, dtype=torch.float32, device=device)
            self.window = make_window(self.win_codes, self.win_scale, wl.win_cap)
        self.pending = torch.zeros(wl.B, 640, dtype=torch.bfloat16, device=device)
        self.ws_append = torch.zeros(csa_workspace_size(OP_APPEND, 0, 0, 0), dtype=torch.uint8, device=device)

    # ---- append ------------------------------------------------------------------
    def append(self, pos0, tok_off, x_bits, y_bits, stream=None):
        """Append host tokens (bf16 bits) through csa_append."""
        T = int(tok_off[-1])
        kv = _bits_to_bf16(x_bits.reshape(T, 512), self.device)
        ix = _bits_to_bf16(y_bits.reshape(T, 128), self.device)
        p0 = _dev(pos0, torch.int32, self.device)
        off = _dev(tok_off, torch.int32, self.device)
        csa_append(self.cache, self.window, p0, off, T, kv, ix, self.pending, self.ws_append, stream)
        return kv, ix, p0, off

    def build_history(self, requests=None, max_tokens_per_call=1 << 18, threads=16):
        """Append each request's history (all tokens before the step's new ones)."""
        wl = self.wl
        reqs = list(range(wl.B)) if requests is None else list(requests)
        units = []                                   # (b, lo, hi) in per-request order
        for b in reqs:
            h = int(wl.hist_len[b])
            for lo in range(0, h, max_tokens_per_call):
                units.append((b, lo, min(h, lo + max_tokens_per_call)))
        calls, cur, cur_t, seen = [], [], 0, set()
        for u in units:
            n = u[2] - u[1]
            if cur and (cur_t + n > max_tokens_per_call or u[0] in seen):
                calls.append(cur)
                cur, cur_t, seen = [], 0, set()
            cur.append(u)
            cur_t += n
            seen.add(u[0])
        if cur:
            calls.append(cur)

        def gen(call):
            parts = []
            for b, lo, hi in call:
                subs = [(b, s, min(hi, s + 4096)) for s in range(lo, hi, 4096)]
                parts.append([wl.tokens(*x) for x in subs])
            return parts

        with ThreadPoolExecutor(max_workers=threads) as ex:
            futs = [ex.submit(gen, c) for c in calls[:2]]
            for i, call in enumerate(calls):
                parts = futs[i].result()
                if i + 2 < len(calls):
                    futs.append(ex.submit(gen, calls[i + 2]))
                pos0 = np.zeros(wl.B, np.int32)
                cnt = np.zeros(wl.B, np.int64)
                xs, ys = [], []
                order = sorted(range(len(call)), key=lambda k: call[k][0])
                for k in order:
                    b, lo, hi = call[k]
                    pos0[b] = lo
                    cnt[b] = hi - lo
                    xs.extend(p[0] for p in parts[k])
                    ys.extend(p[1] for p in parts[k])
                off = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
                self.append(pos0, off, np.concatenate(xs), np.concatenate(ys))
        torch.cuda.synchronize()

    # ---- step --------------------------------------------------------------------------
    def step_inputs(self):
        wl = self.wl
        q_idx, w, q = wl.step_queries()
        x, y = wl.step_tokens()
        s = {
            "q_idx": _bits_to_bf16(q_idx, self.device), "w": _dev(w, torch.float32, self.device),
            "q": _bits_to_bf16(q, self.device),
            "kv_new": _bits_to_bf16(x, self.device), "idx_new": _bits_to_bf16(y, self.device),
            "pos0": _dev(wl.step_pos0, torch.int32, self.device),
            "tok_off": _dev(wl.step_tok_off, torch.int32, self.device),
            "row_req": _dev(wl.row_req, torch.int32, self.device),
            "row_pos": _dev(wl.row_pos, torch.int32, self.device),
        }
        s["rows"] = make_rows(s["row_req"], s["row_pos"], wl.max_entries, int(wl.new_tok.max()))
        s["out"] = torch.empty(wl.R, wl.H, 512, dtype=torch.bfloat16, device=self.device)
        s["lse"] = torch.empty(wl.R, wl.H, dtype=torch.float32, device=self.device)
        s["topk"] = torch.empty(wl.R, 512, dtype=torch.int32, device=self.device)
        s["ws"] = torch.zeros(csa_workspace_size(OP_DECODE, wl.R, wl.max_entries, wl.H), dtype=torch.uint8,
                              device=self.device)
        return s

    def set_compress(self, inputs):
        """Run the step's append with the compressor steps (csa_append_compress);
        inputs: dict of fp32 numpy arrays kv_gamma, idx_gamma, rope_cos, rope_sin
        and eps (see workloads.compress_inputs), or None to switch them off."""
        if inputs is None:
            self.compress = None
            return
        self._compress_dev = {k: (torch.from_numpy(v).to(self.device) if isinstance(v, np.ndarray) else v)
                              for k, v in inputs.items()}
        d = self._compress_dev
        self.compress = make_compress(d["kv_gamma"], d["idx_gamma"], d["eps"], d["rope_cos"], d["rope_sin"])

    def step_append(self, s, stream=None):
        if getattr(self, "compress", None) is not None:
            csa_append_compress(self.cache, self.window, s["pos0"], s["tok_off"], self.wl.R, s["kv_new"],
                                s["idx_new"], self.pending, self.compress, self.ws_append, stream)
            return
        csa_append(self.cache, self.window, s["pos0"], s["tok_off"], self.wl.R, s["kv_new"], s["idx_new"],
                   self.pending, self.ws_append, stream)

    def step(self, s, stream=None, opts=None):
        """The step's append and decode in one csa_step call (csa_step_ex with
        options); the append's device-side faults land in the decode workspace
        s["ws"]."""
        wl = self.wl
        if opts is not None:
            csa_step_ex(self.cache, self.window, s["pos0"], s["tok_off"], wl.R, s["kv_new"], s["idx_new"],
                        self.pending, getattr(self, "compress", None), s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H,
                        s["q"], wl.softmax_scale, s["out"], s["lse"], s["topk"], opts, s["ws"], stream)
            return
        csa_step(self.cache, self.window, s["pos0"], s["tok_off"], wl.R, s["kv_new"], s["idx_new"], self.pending,
                 getattr(self, "compress", None), s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"],
                 wl.softmax_scale, s["out"], s["lse"], s["topk"], s["ws"], stream)

    def step_decode(self, s, stream=None):
        wl = self.wl
        csa_decode(self.cache, self.window, s["rows"], wl.Hi, s["q_idx"], s["w"], wl.H, s["q"],
                   wl.softmax_scale, s["out"], s["lse"], s["topk"], s["ws"], stream)
