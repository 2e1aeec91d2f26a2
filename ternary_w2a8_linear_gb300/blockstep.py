"""Block-step plumbing for hybrid decoding, host side: the verifier's inputs
are prepared on the GPU stream before the host reads the confidence length.

The pages ("BitMTP: When Multi-Token Prediction Meets Low-Bit Large Language
Models", "Methodology in Plain English") describe the decoding policies over
a drafted block and the runtime mechanism this module demonstrates:

* confidence-only decoding commits the first draft and extends the prefix
  through the consecutive drafts whose probability clears a threshold tau
  (0.9 in their main runs);
* hybrid decoding commits that confidence prefix when it is at least a
  minimum length m (the pages do not report m), and otherwise falls back to
  verification;
* M3 enqueues the preparation of the verifier inputs on the GPU stream
  before the host reads the confidence length and decides whether
  verification is needed at all.

Here one block step is: the draft rows' "fast" projection (FP8 activations,
``BITMTP_FLAG_FP8``), the verifier-input preparation (per-row int8
quantisation of the verifier rows, ``bitmtp_linear_quant_act``) enqueued
right behind the asynchronous copy of the drafts' probabilities to pinned
host memory when ``hoist`` is set (so it runs while the host waits for the
copy and decides), the host's decision, and -- only if the hybrid rule asks
for it -- the verifier's "critical" projection (the int8 path on the prepared
codes).  Without ``hoist`` the preparation is enqueued after the decision, on
the critical path.  The drafts' probabilities come from the model's heads,
which are out of scope: the caller provides them as a device vector written
before the step.  Only the library's calls run on the GPU; this module orders
them and makes the host decision.
"""
from __future__ import annotations

import torch

from . import linear as L


def confidence_length(p, tau: float) -> int:
    """Length of the confidence prefix of a drafted block: the first draft is
    always committed; the prefix then extends through the consecutive
    following drafts with probability p[i] >= tau."""
    n = len(p)
    if n == 0:
        return 0
    length = 1
    while length < n and float(p[length]) >= tau:
        length += 1
    return length


def needs_verification(length: int, m_min: int) -> bool:
    """Hybrid decoding: commit the confidence prefix when it is at least
    m_min drafts long, otherwise verify."""
    return length < m_min


class BlockStep:
    """Buffers and CUDA graphs of one block step, built once and replayed.

    draft:  dict(pk, w_scale, N, K, x [D, K] bf16/fp32, y [D, N], p [D] fp32
            device probabilities of the D drafts)
    verify: dict(pk, w_scale, N, K, x [R, K] bf16/fp32 raw verifier rows,
            y [R, N], optional acc [R, N] int32)

    Three graphs, captured on ``stream`` at construction (each call run once
    first, outside the capture): the draft projection followed by the copy of
    the drafts' probabilities to pinned host memory; the verifier-input
    preparation; the verifier projection.  A step replays them in the order
    ``run`` describes, so the host pays one replay per part and the hoisted
    preparation overlaps the host's wait and decision.
    """

    def __init__(self, draft: dict, verify: dict, tau: float = 0.9, m_min: int = 4, stream=None,
                 draft_flags: int = L.FLAG_FP8):
        self.d, self.v = draft, verify
        self.tau, self.m_min = float(tau), int(m_min)
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.draft_flags = draft_flags
        dev = draft["x"].device
        R, K = verify["x"].shape
        self.q = torch.empty((R, K), dtype=torch.int8, device=dev)
        self.a_scale = torch.empty(R, dtype=torch.float32, device=dev)
        self.rowsum = torch.empty(R, dtype=torch.int32, device=dev)
        D = draft["x"].shape[0]
        self.p_host = torch.empty(D, dtype=torch.float32, pin_memory=True)
        self.done = torch.cuda.Event()
        self.ws_d = torch.zeros(L.bitmtp_linear_workspace_bytes(draft["N"], draft["K"], D),
                                dtype=torch.uint8, device=dev)
        self.ws_v = torch.zeros(L.bitmtp_linear_workspace_bytes(verify["N"], verify["K"], R),
                                dtype=torch.uint8, device=dev)
        self._act_d = L.make_act(draft["x"])
        self._out_d = L.make_out(draft["y"])
        self._act_v = L.make_act(self.q, self.a_scale)
        self._out_v = L.make_out(verify["y"], verify.get("acc"))
        # the zero-filled workspaces (and the caller's buffers) before the first call
        self.stream.wait_stream(torch.cuda.current_stream())
        self.g_draft = self._graph(self._draft)
        self.g_prep = self._graph(self._prepare_verifier_inputs)
        # the verifier's graph reads the codes as they are at replay time; the
        # run before its capture sees codes that the preparation just wrote
        self.g_verify = self._graph(self._verify)

    def _graph(self, fn):
        with torch.cuda.stream(self.stream):
            fn()  # first call outside the capture (one-time library set-up)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        return g

    def _cs(self):
        return L._stream(torch.cuda.current_stream())

    def _draft(self):
        d = self.d
        L._check(L.bitmtp_linear_gemm(L._ptr(d["pk"]), float(d["w_scale"]), d["N"], d["K"], d["x"].shape[0],
                                      self._act_d, self._out_d, L._ptr(self.ws_d), self.ws_d.numel(),
                                      self.draft_flags, self._cs()), "draft gemm")
        self.p_host.copy_(d["p"], non_blocking=True)

    def _prepare_verifier_inputs(self):
        x = self.v["x"]
        R, K = x.shape
        L._check(L.bitmtp_linear_quant_act(L._ptr(x), L._act_kind(x), R, K, L._rowmajor(x, "x"), L._ptr(self.q),
                                           K, L._ptr(self.a_scale), L._ptr(self.rowsum), self._cs()), "quant_act")

    def _verify(self):
        v = self.v
        L._check(L.bitmtp_linear_gemm(L._ptr(v["pk"]), float(v["w_scale"]), v["N"], v["K"], v["x"].shape[0],
                                      self._act_v, self._out_v, L._ptr(self.ws_v), self.ws_v.numel(), 0,
                                      self._cs()), "verify gemm")

    def run(self, hoist: bool = True):
        """One block step.  Returns (confidence length, verified).

        The draft graph (projection, then the probabilities' copy) and an
        event; with ``hoist`` the preparation graph right behind them, so it
        runs while the host waits for the event and decides; the host reads
        the probabilities and applies the hybrid rule; only if verification
        is needed the verifier graph (after the preparation graph when not
        hoisted)."""
        with torch.cuda.stream(self.stream):
            self.g_draft.replay()
            self.done.record(self.stream)
            if hoist:
                self.g_prep.replay()
        self.done.synchronize()  # the host reads the drafts' probabilities
        length = confidence_length(self.p_host.tolist(), self.tau)
        verify = needs_verification(length, self.m_min)
        if verify:
            with torch.cuda.stream(self.stream):
                if not hoist:
                    self.g_prep.replay()
                self.g_verify.replay()
        return length, verify
