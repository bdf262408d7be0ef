"""One decode step over a paged KV cache: append the new token, then attend.

``DecodeStep`` owns nothing but the caller's tensors and a workspace; each
method is one or two C-ABI calls (see ``_abi``).  ``run_from_host`` is the
end-to-end form a serving loop uses: the step's per-token inputs arrive in
pinned host memory, are copied to the device, the step runs, and the
attention output is copied back.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi


class DecodeStep:
    """Append + decode for one batch shape.

    Pools are [NB][Hkv][bs][D]: 16-bit (``kv="f16"|"bf16"``) or E4M3 codes
    with fp32 [NB][Hkv] scales (``kv="fp8"``, q/out fp16).
    """

    def __init__(self, *, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
                 num_q_heads, k_scale=None, v_scale=None, split_ctas=0, window=0,
                 early_prologue=False, queries_per_seq=1, workspace=None, early_copies=False):
        self.kv = "fp8" if k_cache.dtype == torch.uint8 else "16"
        self.k_cache, self.v_cache = k_cache, v_cache
        self.k_scale, self.v_scale = k_scale, v_scale
        self.block_tables, self.context_lens = block_tables, context_lens
        self.max_context_len = int(max_context_len)
        self.scale = float(scale)
        self.B = int(block_tables.shape[0])
        self.Hq = int(num_q_heads)
        self.NB, self.Hkv, self.bs, self.D = (int(x) for x in k_cache.shape)
        # query rows per (sequence, kv head) of a decode call: its query tokens
        # (queries_per_seq; the fused step takes one) times the query group
        rows = int(queries_per_seq) * (self.Hq // self.Hkv)
        # more than 8 query rows: two CTAs per SM for every pool type
        self.split_ctas = int(split_ctas) or _abi.pa_decode_default_splits(
            k_cache.dtype if rows <= 8 else torch.float16)
        self.window = int(window)           # sliding window in tokens, 0 for the whole context
        # the attention launch's prologue may overlap the kernel before it on
        # the stream (which must then not write context_lens or block_tables)
        self.early_prologue = bool(early_prologue)
        # PA_DECODE_EARLY_COPIES: the kernels before each call write the pools
        # only in each sequence's last two blocks (the previous step's append)
        self.early_copies = bool(early_copies)
        if self.early_copies and not self.early_prologue:
            raise ValueError("early_copies needs early_prologue")
        # The split-K workspace: zero-filled, left zero-filled by every call.
        # Steps that run one after another on one stream (the slots of a
        # StepPipeline) may share one (``workspace``: a uint8 device tensor of
        # at least pa_decode_workspace_size_rows bytes), which keeps it hot in
        # L2 for all of them.
        need = _abi.pa_decode_workspace_size_rows(self.B, self.Hq, self.D, self.split_ctas, rows)
        if workspace is not None:
            if workspace.numel() * workspace.element_size() < need or workspace.device != k_cache.device:
                raise ValueError(f"workspace too small or on another device: {need} bytes needed")
            self.workspace = workspace
        else:
            self.workspace = _abi.alloc_workspace(self.B, self.Hq, self.D, self.split_ctas,
                                                  k_cache.device, query_rows=rows)
        self._bound = {}     # run_from_staging's bound steps

    def append(self, k_new, v_new, slot_mapping):
        if self.kv == "fp8":
            _abi.pa_cache_append_fp8(k_new, v_new, self.k_cache, self.v_cache, self.k_scale,
                                     self.v_scale, slot_mapping)
        else:
            _abi.pa_cache_append(k_new, v_new, self.k_cache, self.v_cache, slot_mapping)

    def decode(self, q, out):
        if self.kv == "fp8":
            _abi.pa_decode_fp8(out, q, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                               self.block_tables, self.context_lens, self.max_context_len,
                               self.scale, self.split_ctas, self.workspace, window=self.window,
                               early_prologue=self.early_prologue, early_copies=self.early_copies)
        else:
            _abi.pa_decode(out, q, self.k_cache, self.v_cache, self.block_tables,
                           self.context_lens, self.max_context_len, self.scale,
                           self.split_ctas, self.workspace, window=self.window,
                           early_prologue=self.early_prologue, early_copies=self.early_copies)

    def fused(self, q, k_new, v_new, slot_mapping, out, sync=None, copies=None):
        """Append and decode in one launch (slot_mapping must hold each
        sequence's position context_len - 1, as a decode step does); ``sync``
        (an ``_abi.StepSync``) adds the device-side handshake with the copies
        of a serving loop (``StepPipeline``)."""
        if self.kv == "fp8":
            _abi.pa_decode_step_fp8(out, q, k_new, v_new, self.k_cache, self.v_cache,
                                    self.k_scale, self.v_scale, slot_mapping, self.block_tables,
                                    self.context_lens, self.max_context_len, self.scale,
                                    self.split_ctas, self.workspace, window=self.window,
                                    early_prologue=self.early_prologue,
                                    early_copies=self.early_copies, sync=sync,
                                    copies=copies)
        else:
            _abi.pa_decode_step(out, q, k_new, v_new, self.k_cache, self.v_cache, slot_mapping,
                                self.block_tables, self.context_lens, self.max_context_len,
                                self.scale, self.split_ctas, self.workspace, window=self.window,
                                early_prologue=self.early_prologue,
                                early_copies=self.early_copies, sync=sync, copies=copies)
        return out

    @property
    def prefers_fused(self) -> bool:
        """Whether the one-launch step is the faster form for this pool type.

        16-bit pools: yes (on the Qwen2.5-7B batch, 86 us against 98 us for
        append + decode).  E4M3 pools: no; the fused E4M3 kernel runs with
        fewer free registers (three CTAs per SM) and its attention loop loses
        more than the separate append launch costs (760 us against 735 us on
        the 256-sequence E4M3 batch)."""
        return self.kv != "fp8"

    def __call__(self, q, k_new, v_new, slot_mapping, out, fused=None, sync=None):
        """One step; ``fused`` None picks the faster form (``prefers_fused``);
        ``sync`` only with the fused form."""
        if fused is None:
            fused = self.prefers_fused
        if sync is not None and not fused:
            raise ValueError("the device-side handshake needs the fused step")
        if fused:
            return self.fused(q, k_new, v_new, slot_mapping, out, sync=sync)
        self.append(k_new, v_new, slot_mapping)
        self.decode(q, out)
        return out

    def bind(self, q, k_new, v_new, slot_mapping, out, fused=None, stream=None, sync=None):
        """The step on these tensors as a callable with its C-ABI arguments
        checked and marshalled once (``_abi.prepare``), launching on
        ``stream`` (default: the current stream at each call).  Each call
        runs one step; refill the tensors in place between calls (and
        ``sync``'s values, which each call reads)."""
        return _abi.prepare(lambda: self(q, k_new, v_new, slot_mapping, out, fused=fused,
                                         sync=sync), stream)

    def capture(self, q, k_new, v_new, slot_mapping, out, fused=None, stream=None):
        """Record the step into a CUDA graph and return it (``torch.cuda.CUDAGraph``).

        The graph holds the launch(es) with these tensors' addresses: for
        each later step write that step's q, k_new, v_new and slot_mapping
        (and the grown context_lens / block_tables this object was built
        with) into the same tensors, then ``replay()``; ``out`` receives the
        result.  The kernel reads lengths and tables on the device, so one
        graph serves every step while lengths stay within max_context_len.

        Before capturing, the step runs once eagerly on the current stream
        (the library's per-device set-up happens outside the capture).  That
        run is the step itself: it appends the given rows and writes out,
        and a replay with unchanged inputs writes the same bytes again.
        """
        self(q, k_new, v_new, slot_mapping, out, fused=fused)
        torch.cuda.current_stream().synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self(q, k_new, v_new, slot_mapping, out, fused=fused)
        return graph

    def run_from_host(self, host_in: dict, dev_in: dict, host_out, dev_out, fused=None):
        """Copy the step's inputs from pinned host tensors, run it, copy the output back.

        host_in/dev_in map q, k_new, v_new, slot_mapping, block_tables and
        context_lens to same-shaped pinned-host / device tensors (the device
        block_tables and context_lens must be the ones this step was built
        with).  Returns (h2d bytes, d2h bytes).
        """
        h2d = 0
        for k, h in host_in.items():
            dev_in[k].copy_(h, non_blocking=True)
            h2d += h.numel() * h.element_size()
        self(dev_in["q"], dev_in["k_new"], dev_in["v_new"], dev_in["slot_mapping"], dev_out,
             fused=fused)
        host_out.copy_(dev_out, non_blocking=True)
        return h2d, host_out.numel() * host_out.element_size()

    def run_from_staging(self, staging: "StepStaging", host_out, dev_out, fused=None):
        """As ``run_from_host`` with the inputs packed in one ``StepStaging``:
        one host-to-device copy for all of them (this step must have been
        built with the staging's device block_tables and context_lens).  The
        step is bound (``bind``) on first use with a staging and output and
        reused after.  Returns (h2d bytes, d2h bytes)."""
        h2d = staging.upload()
        key = (id(staging), id(dev_out), fused, torch.cuda.current_stream().cuda_stream)
        call = self._bound.get(key)
        if call is None:             # bound once per (staging, output, form, stream)
            d = staging.dev
            call = self.bind(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], dev_out,
                             fused=fused, stream=torch.cuda.current_stream())
            self._bound[key] = call
        call()
        host_out.copy_(dev_out, non_blocking=True)
        return h2d, host_out.numel() * host_out.element_size()


class StepStaging:
    """A decode step's per-step inputs packed back to back (each at a 256-byte
    aligned offset) in one pinned host buffer and one device buffer of the
    same layout.  ``host[name]`` / ``dev[name]`` are views of the two; fill
    the host views, then ``upload()`` moves everything in one copy.  A
    serving loop that uploads its step inputs as one block pays one copy's
    latency instead of one per tensor."""

    def __init__(self, specs: dict, device):
        """specs: name -> (shape, torch dtype)."""
        layout, o = {}, 0
        for name, (shape, dtype) in specs.items():
            n = 1
            for x in shape:
                n *= int(x)
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            layout[name] = (o, tuple(int(x) for x in shape), dtype, nbytes)
            o = (o + nbytes + 255) // 256 * 256
        self.nbytes = max(o, 256)
        self.host_buf = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
        self.dev_buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.host, self.dev = {}, {}
        for name, (off, shape, dtype, nbytes) in layout.items():
            self.host[name] = self.host_buf[off:off + nbytes].view(dtype).view(shape)
            self.dev[name] = self.dev_buf[off:off + nbytes].view(dtype).view(shape)

    def upload(self) -> int:
        """One asynchronous host-to-device copy on the current stream; the bytes copied."""
        self.dev_buf.copy_(self.host_buf, non_blocking=True)
        return self.nbytes


class StepPipeline:
    """Decode steps whose host<->device copies overlap the previous step's
    attention.  ``depth`` stagings (and output buffers) are used in turn:
    uploads run on one copy stream and read-backs on another (on one stream
    the next upload would queue behind the read-back that waits for the
    current step), the steps in order on a compute stream of the pipeline's
    own, with events keeping a staging from being re-uploaded while a step
    still reads it and an output buffer from being rewritten before it is
    read back.  Each slot's step is bound once (``DecodeStep.bind``), and
    the events are made once and recorded again at every use, so a submit
    costs the host a handful of calls.
    Each submit first orders the compute stream after the caller's stream;
    ``finish`` orders the caller's stream after everything submitted.
    Steps built with ``early_prologue`` are fine here: the kernel before a
    step on the compute stream is the previous step's merge, and the upload
    of the step's lengths and tables is ordered before it by an event (a
    full dependency, which the early prologue does not relax).

    ``make_step(staging)`` builds the DecodeStep for one staging (bound to its
    device block_tables and context_lens; the pools are shared, and the steps
    may share one workspace: they run one after another on the compute
    stream).  The caller
    fills ``stagings[k].host`` before ``submit`` uses slot k (``slot()`` says
    which; ``wait_slot_free()`` waits until its last upload has finished)."""

    def __init__(self, make_step, specs: dict, out_shape, out_dtype, device, depth: int = 2,
                 handshake: str = "auto"):
        self.depth = depth
        self.copy = torch.cuda.Stream(device)       # uploads
        self.back = torch.cuda.Stream(device)       # read-backs
        self.compute = torch.cuda.Stream(device)
        self.stagings = [StepStaging(specs, device) for _ in range(depth)]
        self.steps = [make_step(s) for s in self.stagings]
        self.dev_out = [torch.empty(out_shape, dtype=out_dtype, device=device)
                        for _ in range(depth)]
        self.host_out = [torch.empty(out_shape, dtype=out_dtype).pin_memory()
                         for _ in range(depth)]
        self.uploaded = [torch.cuda.Event() for _ in range(depth)]    # the slot's upload done
        self.stepped = [torch.cuda.Event() for _ in range(depth)]     # the slot's step done
        self.read_back = [torch.cuda.Event() for _ in range(depth)]   # its output on the host
        self.calls = {}        # (slot, fused, device handshake) -> the bound step
        self.n = 0
        # Device-side handshake (fused steps): per slot a "ready" word the
        # upload stream sets after the upload, and a "done" word (with the
        # merge launch's CTA count) the step sets when its output is complete;
        # each in its own 32-byte sector.
        self.words = torch.zeros(depth, 3, 8, dtype=torch.int32, device=device)
        self.syncs = []
        for k in range(depth):
            sy = _abi.StepSync()
            sy.ready = self.words[k, 0].data_ptr()
            sy.done = self.words[k, 1].data_ptr()
            sy.done_count = self.words[k, 2].data_ptr()
            self.syncs.append(sy)
        # the word operations of a submit, marshalled once: library entry
        # points with the words' addresses and the streams' handles
        lib = _abi.load()
        self._write_word, self._wait_word = lib.pa_stream_write_value, lib.pa_stream_wait_value
        self._ready_p = [ctypes.c_void_p(self.words[k, 0].data_ptr()) for k in range(depth)]
        self._done_p = [ctypes.c_void_p(self.words[k, 1].data_ptr()) for k in range(depth)]
        self._copy_h = ctypes.c_void_p(self.copy.cuda_stream)
        self._back_h = ctypes.c_void_p(self.back.cuda_stream)
        # the copies of each slot's pipelined step, for the one-call form
        # (pa_decode_step_pipelined): the slot's buffers, the two copy
        # streams and the slot's read-back event (recorded once here so that
        # its handle exists)
        self.copies = []
        for k in range(depth):
            st, io = self.stagings[k], _abi.StepCopies()
            io.host_in, io.dev_in, io.in_bytes = (st.host_buf.data_ptr(), st.dev_buf.data_ptr(),
                                                  st.nbytes)
            io.dev_out, io.host_out = self.dev_out[k].data_ptr(), self.host_out[k].data_ptr()
            io.out_bytes = self.dev_out[k].numel() * self.dev_out[k].element_size()
            io.copy_stream, io.back_stream = self.copy.cuda_stream, self.back.cuda_stream
            self.read_back[k].record(self.back)
            io.reuse_event = self.read_back[k].cuda_event
            io.slot_reused = 0
            self.copies.append(io)
        self.handshake = handshake
        if handshake == "auto":
            try:
                _abi.pa_stream_write_value(self.words[0, 0, :1], 0, self.copy)
                self.handshake = "device"
            except _abi.PAError as e:
                if e.code != _abi.PA_ERR_UNSUPPORTED:
                    raise
                self.handshake = "events"
        self._fresh = True

    def slot(self) -> int:
        return self.n % self.depth

    def wait_slot_free(self):
        """Block the host until the next slot's host buffer may be refilled."""
        if self.n >= self.depth:
            if self.uses_device_handshake():   # the one-call form records only the read-back
                self.read_back[self.slot()].synchronize()
            else:
                self.uploaded[self.slot()].synchronize()

    def _call(self, k, fused, device):
        key = (k, fused, device)
        if key not in self.calls:
            d = self.stagings[k].dev
            if device:   # the whole pipelined step, copies included, in one library call
                st, out = self.steps[k], self.dev_out[k]
                self.calls[key] = _abi.prepare(
                    lambda: st.fused(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], out,
                                     sync=self.syncs[k], copies=self.copies[k]), self.compute)
            else:
                self.calls[key] = self.steps[k].bind(d["q"], d["k_new"], d["v_new"],
                                                     d["slot_mapping"], self.dev_out[k],
                                                     fused=fused, stream=self.compute)
        return self.calls[key]

    def uses_device_handshake(self, fused=None) -> bool:
        """Whether submit(fused) orders its copies by the device-side handshake
        (fused steps, where the driver offers stream memory operations)."""
        if fused is None:
            fused = self.steps[0].prefers_fused
        return self.handshake == "device" and bool(fused)

    def submit(self, fused=None):
        """Upload the next slot's inputs, run its step, read its output back.
        Returns (slot, h2d bytes, d2h bytes); ``host_out[slot]`` holds the
        output once ``read_back[slot]`` has completed."""
        if fused is None:
            fused = self.steps[0].prefers_fused
        if self.uses_device_handshake(fused):
            return self._submit_device(fused)
        k = self.slot()
        reused = self.n >= self.depth
        step = self._call(k, fused, False)
        self.compute.wait_stream(torch.cuda.current_stream())
        if reused:
            self.copy.wait_event(self.stepped[k])         # the slot's last step is done with it
        with torch.cuda.stream(self.copy):
            h2d = self.stagings[k].upload()
        self.uploaded[k].record(self.copy)
        self.compute.wait_event(self.uploaded[k])
        if reused:
            self.compute.wait_event(self.read_back[k])    # the slot's last output was read
        step()
        self.stepped[k].record(self.compute)
        self.back.wait_event(self.stepped[k])
        with torch.cuda.stream(self.back):
            self.host_out[k].copy_(self.dev_out[k], non_blocking=True)
        self.read_back[k].record(self.back)
        self.n += 1
        return k, h2d, self.host_out[k].numel() * self.host_out[k].element_size()

    def _submit_device(self, fused):
        """submit() with the device-side handshake, as one library call
        (pa_decode_step_pipelined): the upload and the ready word on the copy
        stream, the step's kernels alone on the compute stream (the attention
        launch waits on the device for its upload), the wait for the step's
        done word and the read-back on the read-back stream, so consecutive
        steps overlap as they do without copies."""
        k = self.slot()
        seq = (self.n + 1) & 0xffffffff
        step = self._call(k, fused, True)
        if self._fresh:       # order everything after the caller's earlier work, once
            cur = torch.cuda.current_stream()
            for st in (self.compute, self.copy, self.back):
                st.wait_stream(cur)
            self._fresh = False
        sy, io = self.syncs[k], self.copies[k]
        sy.ready_value = seq
        sy.done_value = seq
        io.slot_reused = 1 if self.n >= self.depth else 0
        step()
        self.n += 1
        return k, io.in_bytes, io.out_bytes

    def finish(self):
        """Make the caller's stream wait for every step and copy submitted so far."""
        for st in (self.compute, self.copy, self.back):
            torch.cuda.current_stream().wait_stream(st)
        self._fresh = True
