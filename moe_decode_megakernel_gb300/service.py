"""Binding of the host decode service (include/mk_service.h): argument
marshalling only; the loop, the page allocator and the batching run in
libmk.so, and the GPU step is mk_decode_step plus the library's argmax.

A step function is either a Python callable (tests: it receives numpy views
of the host arrays and fills `next_tokens`) or a GpuStep."""
from __future__ import annotations

import ctypes

import numpy as np

from . import MK_OK, MkError, Model, Sched, _check, lib, last_error

RUNNING, PARKED, FINISHED = 0, 1, 2
FIN_NONE, FIN_LENGTH, FIN_STOP, FIN_CONTEXT, FIN_CANCEL = 0, 1, 2, 3, 4


class MkServiceCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_pages", "page_size", "max_pages", "max_batch")]


class MkSeqInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("state", "finish", "n_ctx", "n_generated", "n_pending",
                                              "n_pages")]


_i32p = ctypes.POINTER(ctypes.c_int32)
TOKEN_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32)
STEP_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, _i32p, _i32p, _i32p, ctypes.c_int32,
                           ctypes.c_int32, _i32p)
_sigs_done = False


def _lib():
    global _sigs_done
    L = lib()
    if not _sigs_done:
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "mk_service_create": (ctypes.c_int, [ctypes.POINTER(MkServiceCfg), vp, vp, ctypes.POINTER(vp)]),
            "mk_service_free": (None, [vp]),
            "mk_service_add": (ctypes.c_int, [vp, i64, _i32p, i32, i32, i32]),
            "mk_service_step": (ctypes.c_int, [vp, ctypes.POINTER(i64), _i32p, i32, _i32p]),
            "mk_service_run": (ctypes.c_int, [vp, i32, vp, vp, _i32p]),
            "mk_service_park": (ctypes.c_int, [vp, i64]),
            "mk_service_resume": (ctypes.c_int, [vp, i64, _i32p, i32]),
            "mk_service_cancel": (ctypes.c_int, [vp, i64]),
            "mk_service_forget": (ctypes.c_int, [vp, i64]),
            "mk_service_query": (ctypes.c_int, [vp, i64, ctypes.POINTER(MkSeqInfo)]),
            "mk_service_pages": (i32, [vp, i64, _i32p, i32]),
            "mk_service_free_pages": (i32, [vp]),
            "mk_service_live": (i32, [vp]),
            "mk_gpu_step_dev_bytes": (sz, [vp, i32, i32]),
            "mk_gpu_step_create": (ctypes.c_int, [vp, ctypes.POINTER(vp), i32, vp, vp, i64, i32, vp, sz, vp,
                                                  sz, vp, ctypes.POINTER(vp)]),
            "mk_gpu_step_free": (None, [vp]),
            "mk_argmax_rows": (ctypes.c_int, [vp, i32, i32, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _sigs_done = True
    return L


def argmax_rows(logits, next_tokens, stream: int = 0) -> None:
    """mk_argmax_rows on device tensors: fp32 [rows][vocab] -> int32 [rows]."""
    rows, vocab = logits.shape
    _check(_lib().mk_argmax_rows(logits.data_ptr(), rows, vocab, next_tokens.data_ptr(), stream))


class GpuStep:
    """mk_gpu_step on torch-owned device memory: the schedules (uploaded
    here), one workspace for all of them, the step's input/output buffer and
    a stream of its own."""

    def __init__(self, model: Model, scheds: list[Sched], k_pool, v_pool, max_pages: int, device="cuda"):
        import torch
        from . import Session
        self.model, self.scheds = model, scheds
        self.sessions = [Session(model, s, device) for s in scheds]  # uploads the lists
        ws = max(s.workspace_bytes() for s in scheds)
        self.workspace = torch.zeros(ws + 256, dtype=torch.uint8, device=device)
        ws_ptr = (self.workspace.data_ptr() + 255) // 256 * 256
        mb = max(s.max_batch for s in scheds)
        nbytes = int(_lib().mk_gpu_step_dev_bytes(model.handle, mb, max_pages))
        self.buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        buf_ptr = (self.buf.data_ptr() + 255) // 256 * 256
        self.k_pool, self.v_pool = k_pool, v_pool
        handles = (ctypes.c_void_p * len(scheds))(*[s.handle.value for s in scheds])
        h = ctypes.c_void_p()
        # a stream of its own (steps are captured as CUDA graphs; the legacy
        # default stream cannot be), after the work that made the weights and pools
        torch.cuda.current_stream(device).synchronize()
        self.stream = torch.cuda.Stream(device)
        st = self.stream.cuda_stream
        _check(_lib().mk_gpu_step_create(model.handle, handles, len(scheds), k_pool.data_ptr(),
                                         v_pool.data_ptr(), k_pool.shape[1], max_pages, ws_ptr, ws, buf_ptr,
                                         nbytes, st, ctypes.byref(h)))
        self.handle = h

    def c_step(self):
        """(function pointer, ctx) for mk_service_create."""
        return ctypes.cast(_lib().mk_gpu_step_run, ctypes.c_void_p), self.handle

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                lib().mk_gpu_step_free(self.handle)
            except Exception:  # interpreter shutdown
                pass
            self.handle = None


class Service:
    """mk_service: admit sequences, step, park/resume/cancel, query."""

    def __init__(self, num_pages: int, page_size: int, max_pages: int, max_batch: int, step):
        self.cfg = MkServiceCfg(num_pages, page_size, max_pages, max_batch)
        if isinstance(step, GpuStep):
            fn, ctx = step.c_step()
            self._keep = step
        else:
            def tramp(_ctx, tok, lens, bt, batch, width, nxt):
                try:
                    t = np.ctypeslib.as_array(tok, shape=(batch,))
                    sl = np.ctypeslib.as_array(lens, shape=(batch,))
                    b = np.ctypeslib.as_array(bt, shape=(batch, width))
                    out = np.ctypeslib.as_array(nxt, shape=(batch,))
                    rc = step(t.copy(), sl.copy(), b.copy(), out)
                    return MK_OK if rc is None else int(rc)
                except Exception:  # an exception cannot cross the C frame
                    import traceback
                    traceback.print_exc()
                    return -1
            self._keep = STEP_FN(tramp)
            fn, ctx = ctypes.cast(self._keep, ctypes.c_void_p), None
        h = ctypes.c_void_p()
        _check(_lib().mk_service_create(ctypes.byref(self.cfg), fn, ctx, ctypes.byref(h)))
        self.handle = h
        n = max_batch
        self._ids = (ctypes.c_int64 * n)()
        self._toks = (ctypes.c_int32 * n)()

    def __del__(self):
        if getattr(self, "handle", None):
            try:
                lib().mk_service_free(self.handle)
            except Exception:  # interpreter shutdown
                pass
            self.handle = None

    def add(self, sid: int, prompt, max_new: int, stop_token: int = -1) -> None:
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        _check(_lib().mk_service_add(self.handle, sid, p.ctypes.data_as(_i32p), p.size, max_new, stop_token))

    def step(self):
        """One step: (rows decoded, [(id, token), ...] sampled)."""
        n = ctypes.c_int32()
        rc = _lib().mk_service_step(self.handle, self._ids, self._toks, self.cfg.max_batch, ctypes.byref(n))
        if rc < 0:
            raise MkError(rc, last_error())
        return rc, [(int(self._ids[i]), int(self._toks[i])) for i in range(n.value)]

    def park(self, sid: int) -> None:
        _check(_lib().mk_service_park(self.handle, sid))

    def resume(self, sid: int, tokens=()) -> None:
        p = np.ascontiguousarray(tokens, dtype=np.int32)
        _check(_lib().mk_service_resume(self.handle, sid, p.ctypes.data_as(_i32p), p.size))

    def cancel(self, sid: int) -> None:
        _check(_lib().mk_service_cancel(self.handle, sid))

    def forget(self, sid: int) -> None:
        _check(_lib().mk_service_forget(self.handle, sid))

    def query(self, sid: int) -> MkSeqInfo:
        info = MkSeqInfo()
        _check(_lib().mk_service_query(self.handle, sid, ctypes.byref(info)))
        return info

    def pages(self, sid: int) -> list[int]:
        buf = (ctypes.c_int32 * self.cfg.max_pages)()
        n = _lib().mk_service_pages(self.handle, sid, buf, self.cfg.max_pages)
        if n < 0:
            raise MkError(n, last_error())
        return [int(buf[i]) for i in range(n)]

    @property
    def free_pages(self) -> int:
        return int(_lib().mk_service_free_pages(self.handle))

    @property
    def live(self) -> int:
        return int(_lib().mk_service_live(self.handle))

    def run(self, max_steps: int = (1 << 31) - 1, on_token=None) -> dict[int, list[int]]:
        """mk_service_run: the library steps until nothing can run (or
        max_steps), streaming each sampled token to on_token(id, token);
        returns the sampled tokens per id."""
        out: dict[int, list[int]] = {}

        def cb(_ctx, sid, tok):
            out.setdefault(int(sid), []).append(int(tok))
            if on_token is not None:
                on_token(int(sid), int(tok))
        fn = TOKEN_FN(cb)
        steps = ctypes.c_int32()
        rc = _lib().mk_service_run(self.handle, max_steps, ctypes.cast(fn, ctypes.c_void_p), None,
                                   ctypes.byref(steps))
        if rc != MK_OK:
            raise MkError(rc, last_error())
        self.last_run_steps = steps.value
        return out
