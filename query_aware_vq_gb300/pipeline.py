"""One step of the A2ATS hot path, composed from the C-ABI calls.

The order is the one the pages' cache wrapper runs every step (v0.39.0 page,
"How it works"; deploy-preview page, "Per-step re-rotation" and "Query-aware
VQ (Eq. 13-18)"), with the calibration of H and L in front:

  1. H = E[q^T q] + ridge I            a2ats_query_second_moment
  2. L = chol(H)                       a2ats_cholesky_factor
  3. k~ = windowed RoPE of the cache   a2ats_windowed_rope  } one pass:
  4. retrieval split, proxy query k~_t a2ats_select_retrieval_set  } ..._rotated
  5. retrieval rows: H-weighted rule   a2ats_h_weighted_assign (RoPE fused)
     (or the cosine blend when no H is calibrated)
  6. bulk rows: plain nearest centroid a2ats_h_weighted_assign, L = identity

Steps 4-6 apply the windowed RoPE on the fly in fp32 to the pre-RoPE keys, so
their decisions are taken on the unrounded rotated keys; step 3 writes the
rotated cache in the storage dtype for the attention that follows.  Steps 3
and 4 run as one call (a2ats_select_retrieval_set_rotated) that reads the
pre-RoPE cache once.

The routing is computed as two halves at the same time.  The caller's
stream assigns every row by the bulk rule (plain VQ needs neither the split
nor L) and a second stream the retrieval rows by the retrieval rule into a
buffer of its own; the caller's stream then waits for the second and copies
the retrieval rows' codes over the bulk ones (a2ats_copy_retrieval_rows),
which gives exactly step 5 on the retrieval rows and step 6 on the others.

By default (fused=True) steps 3, 4 and 6 are one call on the caller's
stream, a2ats_rope_split_plain_assign: with far_offset = 0 the keys outside
the RoPE window are their own k~, so the pass of the tensor-core assignment
over them also copies them out and scores them for the split.  The split
itself runs on the second stream (on a third while the second calibrates),
beside the window rows of step 6 on the caller's stream; the call records an
event once it is written, and the second stream starts the retrieval rule
there.  With fused=False the second stream runs steps 3-4 itself, beside
step 6.

Steps 1-2 may also run once, ahead of the steps that reuse their L
(A2ATSStep.calibrate), as the pages do when H is calibrated offline.

All buffers are allocated once in the constructor; a step allocates nothing.
"""
from __future__ import annotations

import torch

from . import (a2ats_append_rows, a2ats_cholesky_factor, a2ats_copy_retrieval_rows,
               a2ats_h_weighted_assign,
               a2ats_query_aware_assign, a2ats_query_second_moment,
               a2ats_rope_split_plain_assign, a2ats_select_retrieval_set,
               a2ats_select_retrieval_set_rotated, a2ats_subvector_assign,
               a2ats_subvector_query_aware_assign, a2ats_windowed_rope, library)


class A2ATSStep:
    def __init__(self, B: int, H: int, N: int, d: int, K: int, dtype: torch.dtype, *,
                 window: int, fraction: float, rope_base: float, far_offset: int = 0,
                 M: int = 0, ridge: float = 1e-4, beta: float = 0.5, interleaved: bool = False,
                 fused: bool = True, device="cuda"):
        self.B, self.H, self.N, self.d, self.K, self.M = B, H, N, d, K, M
        self.fused = fused
        self.dtype, self.fraction, self.ridge, self.beta = dtype, fraction, ridge, beta
        self.rope = dict(window=window, far_offset=far_offset, rope_base=rope_base,
                         interleaved=interleaved)
        dev = torch.device(device)
        lib = library()
        self.k_tilde = torch.empty((B, H, N, d), dtype=dtype, device=dev)
        self.perm = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.count = torch.empty((B, H), dtype=torch.int32, device=dev)
        self.codes = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.codes_retrieval = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.Hm = torch.empty((H, d, d), dtype=torch.float32, device=dev)
        self.L = torch.empty((H, d, d), dtype=torch.float32, device=dev)
        self.info = torch.empty((H,), dtype=torch.int32, device=dev)
        ws = max(lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K),
                 lib.a2ats_query_aware_assign_workspace_size(B, H, N, d, K),
                 lib.a2ats_rope_split_plain_assign_workspace_size(B, H, N, d, K))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        # the split has its own workspace, so the bulk call's codebook side
        # survives from one step to the next
        self.split_workspace = torch.empty(
            lib.a2ats_select_retrieval_set_workspace_size(B, H, N, d), dtype=torch.uint8,
            device=dev)
        # the second stream (calibration, then the retrieval rows) and its
        # own workspace, so that it can run beside the caller's stream
        side = max(lib.a2ats_query_second_moment_workspace_size(H, max(M, 1), d),
                   lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K),
                   lib.a2ats_query_aware_assign_workspace_size(B, H, N, d, K))
        self.side_workspace = torch.empty(side, dtype=torch.uint8, device=dev)
        self.side_stream = torch.cuda.Stream(device=dev)
        # the split's stream while the second one calibrates
        self.split_stream = torch.cuda.Stream(device=dev)
        self.calibrated = False
        self._inputs_ready = torch.cuda.Event()
        self._side_done = torch.cuda.Event()
        # recorded by the library through its handle, which the first record
        # creates
        self._split_done = torch.cuda.Event()
        self._split_done.record(torch.cuda.current_stream(dev))

    @staticmethod
    def _stage(events, name, on, fn, *a, **kw):
        if events is None:
            return fn(*a, stream=on, **kw)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(on)
        r = fn(*a, stream=on, **kw)
        e1.record(on)
        events.setdefault(name, []).append((e0, e1))
        return r

    def calibrate(self, queries=None, h_given=None, stream=None, events=None):
        """H = E[q^T q] + ridge I from queries [H, M, d] (or h_given [H, d, d]
        fp32 as is) and its Cholesky factor, kept in self.Hm / self.L / self.info
        for the steps that follow (the pages calibrate H once per layer, ahead
        of decoding).  Runs on `stream`."""
        st = stream if stream is not None else torch.cuda.current_stream()
        if queries is not None:
            self._stage(events, "second_moment", st, a2ats_query_second_moment, queries,
                        self.ridge, out=self.Hm, workspace=self.side_workspace)
            h_given = self.Hm
        if h_given is None:
            raise ValueError("calibrate needs queries or h_given")
        self._stage(events, "cholesky", st, a2ats_cholesky_factor, h_given, out=self.L,
                    info=self.info)
        self.calibrated = True
        return self

    def __call__(self, keys, codebook, queries=None, h_given=None, lengths=None, stream=None,
                 events=None, calibrated=False, reuse_codebook=False):
        """keys [B, H, N, d] pre-RoPE; codebook [H, K, d].  The retrieval rows
        take the H-weighted rule with an L calibrated inside the step from
        queries [H, M, d] (or h_given [H, d, d] fp32), or, with
        calibrated=True, the L of an earlier calibrate(); with neither, the
        cosine blend.  reuse_codebook=True takes the codebook side of both
        assignments (the transform by L, its norms and planes) from the
        previous step, which must have had the same codebook, L and shapes
        (the codebook and L are per-layer constants).  Every output is
        complete, in the order of `stream`, when the call's work on `stream`
        is.  events: optional dict; each stage appends a (start, end) CUDA
        event pair recorded around its call on the stream that runs it
        (stages on the two streams overlap)."""
        ws, sws = self.workspace, self.side_workspace
        st = stream if stream is not None else torch.cuda.current_stream()
        side = self.side_stream

        def stage(name, on, fn, *a, **kw):
            return self._stage(events, name, on, fn, *a, **kw)

        self._inputs_ready.record(st)
        side.wait_event(self._inputs_ready)
        L = None
        if queries is not None or h_given is not None:
            self.calibrate(queries, h_given, stream=side, events=events)
            L = self.L
        elif calibrated:
            if not getattr(self, "calibrated", False):
                raise ValueError("calibrated=True before any calibrate()")
            L = self.L
        in_step = queries is not None or h_given is not None
        if self.fused:
            # caller's stream: steps 3, 4 and 6 in one call; the second
            # stream waits for the split only
            stage("rope_split_bulk", st, a2ats_rope_split_plain_assign, keys, codebook, None,
                  self.fraction, rope=self.rope, lengths=lengths, out=self.k_tilde,
                  perm=self.perm, count=self.count, codes=self.codes, reuse=reuse_codebook,
                  split_done=self._split_done,
                  split_stream=self.split_stream if in_step else side, workspace=ws)
            side.wait_event(self._split_done)
        else:
            # second stream: steps 3-4 in one pass over the pre-RoPE cache
            stage("rope_and_split", side, a2ats_select_retrieval_set_rotated, keys, None,
                  self.fraction, rope=self.rope, lengths=lengths, out=self.k_tilde,
                  perm=self.perm, count=self.count, workspace=self.split_workspace)
        # second stream: the retrieval rows into a buffer of their own
        if L is not None:
            stage("assign_retrieval", side, a2ats_h_weighted_assign, keys, codebook, L,
                  lengths=lengths, rope=self.rope, rows="retrieval", perm=self.perm,
                  count=self.count, codes=self.codes_retrieval, workspace=sws,
                  reuse=reuse_codebook and not in_step)
        else:
            # no calibrated H: the cosine blend against the same proxy query
            # (the key at t after windowed RoPE) the split used
            stage("assign_retrieval", side, a2ats_query_aware_assign, keys, codebook, None,
                  self.beta, lengths=lengths, rope=self.rope, rows="retrieval", perm=self.perm,
                  count=self.count, codes=self.codes_retrieval, workspace=sws)
        self._side_done.record(side)
        if not self.fused:
            # caller's stream: the bulk rule over every row (it needs no
            # split)
            stage("assign_bulk", st, a2ats_h_weighted_assign, keys, codebook, None,
                  lengths=lengths, rope=self.rope, rows="all", codes=self.codes, workspace=ws,
                  reuse=reuse_codebook)
        # the retrieval rows' codes over the bulk ones
        st.wait_event(self._side_done)
        stage("route", st, a2ats_copy_retrieval_rows, self.codes_retrieval, self.codes,
              self.perm, self.count, lengths=lengths)
        return self

    def capture(self, keys, codebook, **kw):
        """One step, with the same arguments as a call, captured into a CUDA
        graph (both streams: the second forks from and joins the capturing
        stream through events).  Every replay runs that step again on the same
        buffers; the inputs may be refilled in place between replays.  The
        call warms the step up once on a side stream before capturing."""
        s = torch.cuda.Stream(device=keys.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self(keys, codebook, **kw)
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self(keys, codebook, **kw)
        return graph


class A2ATSDecodeStep:
    """One decode step over a batch of growing caches (v0.39.0 page, "How it
    works", with one incoming key per (sequence, head)):

      1. append the new pre-RoPE keys at position len[b]   a2ats_append_rows
      2. windowed RoPE of the whole cache against the new
         decode position (the per-step re-rotation), and
      3. the retrieval split of every cached key, proxy
         query = the new key after windowed RoPE, in one
         pass over the cache                               a2ats_select_retrieval_set_rotated
      4. the new keys assigned by the cosine blend against
         that proxy (each new key is its own query)        a2ats_query_aware_assign
         (or by the H-weighted rule when L is given)

    cache [B, H, Ncap, d] and lengths [B] int32 are updated in place; the
    rotated cache, split and codes are written to buffers allocated once."""

    def __init__(self, B: int, H: int, N: int, d: int, K: int, dtype: torch.dtype, *,
                 window: int, fraction: float, rope_base: float, beta: float,
                 far_offset: int = 0, interleaved: bool = False, device="cuda"):
        self.fraction, self.beta = fraction, beta
        self.rope = dict(window=window, far_offset=far_offset, rope_base=rope_base,
                         interleaved=interleaved)
        dev = torch.device(device)
        lib = library()
        self.k_tilde = torch.empty((B, H, N, d), dtype=dtype, device=dev)
        self.perm = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.count = torch.empty((B, H), dtype=torch.int32, device=dev)
        self.codes = torch.full((B, H, N), -1, dtype=torch.int32, device=dev)
        # the split's scratch and the assignment's (which keeps the codebook
        # side between steps) in workspaces of their own
        self.workspace = torch.empty(lib.a2ats_select_retrieval_set_workspace_size(B, H, N, d),
                                     dtype=torch.uint8, device=dev)
        ws = max(lib.a2ats_query_aware_assign_workspace_size(B, H, N, d, K),
                 lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K))
        self.assign_workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def __call__(self, cache, lengths, new_keys, codebook, L=None, stream=None, events=None,
                 reuse_codebook=False):
        """reuse_codebook=True takes the codebook side (decoded centroids,
        norms; with L its transform and planes) that the previous call built:
        the caller guarantees the same codebook (and L) as that call."""
        st = stream if stream is not None else torch.cuda.current_stream()
        ws, wa = self.workspace, self.assign_workspace

        def stage(name, fn, *a, **kw):
            if events is None:
                return fn(*a, **kw)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            r = fn(*a, **kw)
            e1.record(st)
            events.setdefault(name, []).append((e0, e1))
            return r

        stage("append", a2ats_append_rows, cache, lengths, new_keys, stream=st)
        stage("rope_and_split", a2ats_select_retrieval_set_rotated, cache, None, self.fraction,
              rope=self.rope, lengths=lengths, out=self.k_tilde, perm=self.perm,
              count=self.count, workspace=ws, stream=st)
        if L is not None:
            stage("assign_new", a2ats_h_weighted_assign, cache, codebook, L, lengths=lengths,
                  rope=self.rope, rows="last", codes=self.codes, workspace=wa, stream=st,
                  reuse=reuse_codebook)
        else:
            stage("assign_new", a2ats_query_aware_assign, cache, codebook, None, self.beta,
                  lengths=lengths, rope=self.rope, rows="last", codes=self.codes, workspace=wa,
                  stream=st, reuse=reuse_codebook)
        return self


class A2ATSSubvectorStep:
    """The pages' wrapper defaults: sub-vector (product) VQ of keys and
    values (v0.39.0 page, configuration a2ats_sub_dim = 8 and
    a2ats_codebook_bits = 8, "How it works" steps 1-5; the API page's
    functions take [N, d] sub-vectors), composed from the C-ABI calls:

      1. k~ = windowed RoPE of the cache, fp32 (the rotation
         pairs elements across sub-vectors, so it runs on
         the whole head first)                                 a2ats_windowed_rope
      2. the retrieval split over tokens (full-width cosine
         with the proxy query k~_t)                            a2ats_select_retrieval_set
      3. every token's sub-vectors: plain nearest centroid     a2ats_h_weighted_assign, L = I
      4. the retrieval tokens' sub-vectors: the H-weighted
         rule with the sub_dim x sub_dim factor L               a2ats_h_weighted_assign
      5. routed by copy over the sub-vector rows               a2ats_copy_retrieval_rows
      6. values' sub-vectors: plain nearest centroid, no RoPE
         and no retrieval preference ("How it works" step 5)   a2ats_h_weighted_assign, L = I

    By default (dedicated=True) steps 3-6 are two calls of
    a2ats_subvector_assign (one pass over the rotated keys applying each
    token's rule from the split, then the values); dedicated=False runs the
    composition listed above, with the same results up to near-ties.  With
    L = None the dedicated path gives the retrieval tokens the page's
    wrapper rule for a cache without a calibrated H: the cosine blend with
    `beta` against the proxy query k~_t, slice by slice
    (a2ats_subvector_query_aware_assign).

    A token of width d is d / sub_dim sub-vector rows; sub-vector row
    j * G + g of a (b, h) is elements g * sub_dim .. of token j (G = d /
    sub_dim).  Codebooks are [H, K, sub_dim] (a table shared by the heads is
    passed once per head).  codes_k and codes_v are [B, H, N, G] int32.
    Buffers are allocated once in the constructor."""

    def __init__(self, B: int, H: int, N: int, d: int, sub_dim: int, K: int, dtype, *,
                 window: int, fraction: float, rope_base: float, interleaved: bool = False,
                 dedicated: bool = True, beta: float = 0.5, device="cuda"):
        if sub_dim < 8 or d % sub_dim:
            raise ValueError("sub_dim must divide d and be at least 8")
        if dedicated and sub_dim not in (8, 16):
            raise ValueError("the sub-vector kernel takes sub_dim 8 or 16")
        self.dedicated = dedicated
        self.beta = beta
        self.B, self.H, self.N, self.d, self.s, self.K = B, H, N, d, sub_dim, K
        self.G = d // sub_dim
        self.fraction = fraction
        self.rope = dict(window=window, far_offset=0, rope_base=rope_base,
                         interleaved=interleaved)
        dev = torch.device(device)
        lib = library()
        G, NG = self.G, N * self.G
        self.k_tilde = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.perm = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.count = torch.empty((B, H), dtype=torch.int32, device=dev)
        self.sub_perm = torch.empty((B, H, N, G), dtype=torch.int32, device=dev)
        self.sub_count = torch.empty((B, H), dtype=torch.int32, device=dev)
        self.sub_len = torch.empty((B,), dtype=torch.int32, device=dev)
        self._g = torch.arange(G, dtype=torch.int32, device=dev)
        self.codes_k = torch.empty((B, H, N, G), dtype=torch.int32, device=dev)
        self.codes_ret = torch.empty((B, H, N, G), dtype=torch.int32, device=dev)
        self.codes_v = torch.empty((B, H, N, G), dtype=torch.int32, device=dev)
        ws = max(lib.a2ats_h_weighted_assign_workspace_size(B, H, NG, sub_dim, K),
                 lib.a2ats_select_retrieval_set_workspace_size(B, H, N, d),
                 lib.a2ats_subvector_assign_workspace_size(B, H, N, d, sub_dim, K),
                 lib.a2ats_subvector_query_aware_assign_workspace_size(B, H, N, d, sub_dim, K))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def __call__(self, keys, values, codebook_k, codebook_v, L, lengths=None, stream=None):
        """keys, values [B, H, N, d] (keys pre-RoPE); codebook_k [H, K, sub_dim]
        fp32 (the rotated keys are fp32), codebook_v [H, K, sub_dim] in the
        values' dtype; L [H, sub_dim, sub_dim] the factor of the sub-vector
        H, or None (the dedicated path then takes the cosine blend);
        lengths [B] int32 or None."""
        st = stream if stream is not None else torch.cuda.current_stream()
        B, H, N, G, s = self.B, self.H, self.N, self.G, self.s
        ws = self.workspace
        if self.dedicated:
            # steps 3-6 in the sub-vector kernel: both rules in one pass over
            # the rotated keys (the split read from perm / count), then the
            # values
            a2ats_windowed_rope(keys, lengths=lengths, out=self.k_tilde, stream=st, **self.rope)
            a2ats_select_retrieval_set(self.k_tilde, None, self.fraction, lengths=lengths,
                                       perm=self.perm, count=self.count, workspace=ws, stream=st)
            if L is not None:
                a2ats_subvector_assign(self.k_tilde, codebook_k, s, L, lengths=lengths,
                                       perm=self.perm, count=self.count, codes=self.codes_k,
                                       workspace=ws, stream=st)
            else:
                # no calibrated H: the wrapper's cosine blend with the proxy
                # query k~_t, slice by slice
                a2ats_subvector_query_aware_assign(self.k_tilde, codebook_k, s, None, self.beta,
                                                   lengths=lengths, perm=self.perm,
                                                   count=self.count, codes=self.codes_k,
                                                   workspace=ws, stream=st)
            a2ats_subvector_assign(values, codebook_v, s, None, lengths=lengths,
                                   codes=self.codes_v, workspace=ws, stream=st)
            return self
        with torch.cuda.stream(st):
            if lengths is None:
                self.sub_len.fill_(N * G)
            else:
                torch.mul(lengths, G, out=self.sub_len)
            a2ats_windowed_rope(keys, lengths=lengths, out=self.k_tilde, stream=st, **self.rope)
            a2ats_select_retrieval_set(self.k_tilde, None, self.fraction, lengths=lengths,
                                       perm=self.perm, count=self.count, workspace=ws, stream=st)
            # sub-vector rows of the retrieval tokens: j * G + g for the
            # token-level split (both halves stay ascending)
            self.sub_perm.copy_(self.perm.unsqueeze(-1).expand(B, H, N, G))
            self.sub_perm.mul_(G).add_(self._g)
            torch.mul(self.count, G, out=self.sub_count)
            ksub = self.k_tilde.view(B, H, N * G, s)
            kc = self.codes_k.view(B, H, N * G)
            a2ats_h_weighted_assign(ksub, codebook_k, None, lengths=self.sub_len, rows="all",
                                    codes=kc, workspace=ws, stream=st)
            a2ats_h_weighted_assign(ksub, codebook_k, L, lengths=self.sub_len, rows="retrieval",
                                    perm=self.sub_perm.view(B, H, N * G), count=self.sub_count,
                                    codes=self.codes_ret.view(B, H, N * G), workspace=ws,
                                    stream=st)
            a2ats_copy_retrieval_rows(self.codes_ret.view(B, H, N * G), kc,
                                      self.sub_perm.view(B, H, N * G), self.sub_count,
                                      lengths=self.sub_len, stream=st)
            vsub = values.reshape(B, H, N * G, s)
            a2ats_h_weighted_assign(vsub, codebook_v, None, lengths=self.sub_len, rows="all",
                                    codes=self.codes_v.view(B, H, N * G), workspace=ws,
                                    stream=st)
        return self
