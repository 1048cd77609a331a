"""Python binding of the GB300 decode megakernel's C ABI (include/mk.h).

Argument marshalling only: every step of the decode path runs in libmk.so's
CUDA kernels.  PyTorch is used for device memory and streams (tensors are
passed to the C ABI as raw pointers).  If libmk.so has not been built the
import of the compute entry points fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

MK_OK, MK_ERR_ARG, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_UNSUPPORTED, MK_ERR_DEVICE = 0, -1, -2, -3, -4, -5
MK_WAVES_DEFAULT, MK_WAVES_INTERLEAVED, MK_WAVES_ATTN_FIRST = 0, 1, 2

# opcodes (field 0 of a task descriptor)
OPS = {0: "NOP", 1: "RESID_NORM", 2: "QKV_PROJ", 3: "O_PROJ", 4: "FFN_UPGATE_ACT", 5: "FFN_DOWN",
       6: "LM_HEAD", 7: "ATTN_DECODE", 8: "ATTN_COMBINE", 9: "ATTN_DRAIN", 10: "ROUTER_GEMM",
       11: "ROUTER_TOPK", 12: "ROUTE_FINALIZE", 13: "MOE_GATHER", 14: "MOE_UPGATE_ACT_DRAIN",
       15: "MOE_DOWN_DRAIN", 16: "MOE_COMBINE"}
F_OP, F_LAYER, F_WAIT0, F_TGT0, F_WAIT1, F_TGT1, F_SIG0, F_SIG1, F_A0, F_TASK = 0, 1, 2, 3, 4, 5, 6, 7, 8, 24


class MkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


class MkConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "hidden", "n_q", "n_kv", "head_dim",
                                              "n_experts", "top_k", "inter", "vocab", "page_size",
                                              "window", "full_period")] + \
               [("rope_base", ctypes.c_float), ("eps", ctypes.c_float), ("expert_fp8", ctypes.c_int32),
                                                                        ("expert_fp4", ctypes.c_int32)]


class MkWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("embedding", "w_qkv", "w_o", "w_router",
                                               "router_bias", "w_gate", "w_up", "w_down",
                                               "norm_gamma", "final_gamma", "w_lm", "w_gate_scale",
                                               "w_up_scale", "w_down_scale", "w_gate_bscale",
                                               "w_up_bscale", "w_down_bscale")]


class MkSchedOpts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_sms", "wave_order", "attn_split_pages",
                                              "attn_claimers", "moe_claimers", "qkv_tile_rows",
                                              "o_tile_rows", "lm_tile_rows", "fuse_finalize",
                                              "fuse_moe_combine", "explicit_gather",
                                              "trace_hidden", "watchdog_ms", "trace", "moe_queue", "moe_static",
                                              "fuse_routing", "fuse_norm_qkv", "attn_static", "moe_balance",
                                              "combine_per_head", "placement", "attn_sms", "trace_queue")]


_lib = None


def lib():
    """The loaded libmk.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "mk_load_model": (ctypes.c_int, [ctypes.POINTER(MkConfig), ctypes.POINTER(MkWeights),
                                             ctypes.POINTER(vp)]),
            "mk_free_model": (None, [vp]),
            "mk_default_sched_opts": (None, [ctypes.POINTER(MkSchedOpts)]),
            "mk_build_tasks": (ctypes.c_int, [vp, i32, i32, ctypes.POINTER(MkSchedOpts),
                                              ctypes.POINTER(vp)]),
            "mk_free_sched": (None, [vp]),
            "mk_sched_bytes": (sz, [vp]),
            "mk_sched_upload": (ctypes.c_int, [vp, vp, sz, vp]),
            "mk_workspace_bytes": (sz, [vp]),
            "mk_decode_step": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, vp, vp, i64, vp, sz, vp,
                                              vp]),
            "mk_check_step": (ctypes.c_int, [vp, vp, vp]),
            "mk_check_inputs": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i64]),
            "mk_decode_step_static_ws": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, vp, vp, i64, vp,
                                                        vp]),
            "mk_last_error": (ctypes.c_char_p, []),
            "mk_workspace_offset": (i64, [vp, ctypes.c_char_p]),
            "mk_sched_num_sms": (i32, [vp]),
            "mk_sched_num_tasks": (i32, [vp, i32]),
            "mk_sched_get_task": (ctypes.c_int, [vp, i32, i32, ctypes.POINTER(i32)]),
            "mk_sched_set_task": (ctypes.c_int, [vp, i32, i32, ctypes.POINTER(i32)]),
            "mk_sched_num_barriers": (i32, [vp]),
            "mk_sched_validate": (ctypes.c_int, [vp]),
            "mk_sched_simulate": (ctypes.c_int, [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                                 ctypes.c_uint64]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().mk_last_error().decode()


def _check(rc: int) -> None:
    if rc != MK_OK:
        raise MkError(rc, last_error())


def _i32p(a):
    import numpy as np
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


# ---------------------------------------------------------------- handles

class Model:
    """mk_load_model: the shape plus the caller's device weight pointers."""

    def __init__(self, cfg: MkConfig, weights: MkWeights, keepalive=None):
        self.cfg = cfg
        self.weights = weights
        self._keep = keepalive
        h = ctypes.c_void_p()
        _check(lib().mk_load_model(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.mk_free_model(self.handle)
            self.handle = None


def default_sched_opts(**kw) -> MkSchedOpts:
    o = MkSchedOpts()
    lib().mk_default_sched_opts(ctypes.byref(o))
    for k, v in kw.items():
        if not hasattr(o, k):
            raise KeyError(k)
        setattr(o, k, int(v))
    return o


class Sched:
    """mk_build_tasks: validated per-SM task lists (host), uploaded on demand."""

    def __init__(self, model: Model, max_batch: int, max_ctx: int, opts: MkSchedOpts | None = None):
        self.model = model
        self.max_batch, self.max_ctx = max_batch, max_ctx
        self.opts = opts if opts is not None else default_sched_opts()
        h = ctypes.c_void_p()
        _check(lib().mk_build_tasks(model.handle, max_batch, max_ctx, ctypes.byref(self.opts),
                                    ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.mk_free_sched(self.handle)
            self.handle = None

    # sizes and upload
    def sched_bytes(self) -> int:
        return int(lib().mk_sched_bytes(self.handle))

    def workspace_bytes(self) -> int:
        return int(lib().mk_workspace_bytes(self.handle))

    def upload(self, dev_ptr: int, nbytes: int, stream: int = 0) -> None:
        _check(lib().mk_sched_upload(self.handle, dev_ptr, nbytes, stream))

    def workspace_offset(self, name: str) -> int:
        return int(lib().mk_workspace_offset(self.handle, name.encode()))

    # inspection
    @property
    def num_sms(self) -> int:
        return int(lib().mk_sched_num_sms(self.handle))

    def num_tasks(self, sm: int) -> int:
        return int(lib().mk_sched_num_tasks(self.handle, sm))

    def get_task(self, sm: int, idx: int):
        import numpy as np
        d = np.zeros(32, np.int32)
        _check(lib().mk_sched_get_task(self.handle, sm, idx,
                                       d.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return d

    def set_task(self, sm: int, idx: int, desc) -> None:
        d, p = _i32p(desc)
        _check(lib().mk_sched_set_task(self.handle, sm, idx, p))

    def num_barriers(self) -> int:
        return int(lib().mk_sched_num_barriers(self.handle))

    def validate(self) -> None:
        _check(lib().mk_sched_validate(self.handle))

    def check_inputs(self, tokens, seq_lens, block_tables, num_pages: int) -> None:
        """mk_check_inputs on host arrays (tokens may be None): raises MkError
        (MK_ERR_ARG) for inputs the step would refuse, before any launch."""
        import numpy as np
        sl, slp = _i32p(seq_lens)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        tp = _i32p(tokens)[1] if tokens is not None else None
        _check(lib().mk_check_inputs(self.handle, tp, slp, bt.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                     sl.size, bt.shape[1], num_pages))

    def simulate(self, seq_lens, routing=None, seed: int = 0) -> None:
        sl, slp = _i32p(seq_lens)
        if routing is not None:
            r, rp = _i32p(routing)
        else:
            rp = None
        _check(lib().mk_sched_simulate(self.handle, sl.size, slp, rp, seed))


def decode_step(model: Model, sched: Sched, last_tokens: int, seq_lens: int, block_tables: int,
                batch: int, max_pages: int, k_pool: int, v_pool: int, num_pages: int,
                workspace: int, workspace_bytes: int, logits: int, stream: int = 0) -> None:
    """mk_decode_step on raw device pointers (see include/mk.h)."""
    _check(lib().mk_decode_step(model.handle, sched.handle, last_tokens, seq_lens, block_tables,
                                batch, max_pages, k_pool, v_pool, num_pages, workspace,
                                workspace_bytes, logits, stream))


def decode_step_static_ws(model: Model, sched: Sched, last_tokens: int, seq_lens: int,
                          block_tables: int, batch: int, max_pages: int, k_pool: int, v_pool: int,
                          num_pages: int, logits: int, stream: int = 0) -> None:
    """mk_decode_step_static_ws: the decode step on the library's built-in
    8 MiB workspace, for callers that cannot allocate device memory (see
    include/mk.h for its sharing rules)."""
    _check(lib().mk_decode_step_static_ws(model.handle, sched.handle, last_tokens, seq_lens,
                                          block_tables, batch, max_pages, k_pool, v_pool, num_pages,
                                          logits, stream))


def check_step(sched: Sched, workspace: int, stream: int = 0) -> None:
    """mk_check_step: waits for the stream, raises MkError on a device failure."""
    _check(lib().mk_check_step(sched.handle, workspace, stream))


class Session:
    """Owns the device copies a step needs (task lists and workspace) as torch
    tensors and calls decode_step with the caller's tensors."""

    def __init__(self, model: Model, sched: Sched, device="cuda"):
        import torch
        self.model, self.sched = model, sched
        self.sched_buf = torch.empty(sched.sched_bytes() + 128, dtype=torch.uint8, device=device)
        p = self.sched_buf.data_ptr()
        self._sched_ptr = (p + 127) // 128 * 128
        sched.upload(self._sched_ptr, sched.sched_bytes(), torch.cuda.current_stream().cuda_stream)
        self.ws_bytes = sched.workspace_bytes()
        self.workspace = torch.zeros(self.ws_bytes + 256, dtype=torch.uint8, device=device)
        self.ws_ptr = (self.workspace.data_ptr() + 255) // 256 * 256
        self.ws_base = self.ws_ptr - self.workspace.data_ptr()

    def step(self, tokens, seq_lens, block_tables, k_pool, v_pool, logits, stream=None) -> None:
        import torch
        st = (stream or torch.cuda.current_stream()).cuda_stream
        decode_step(self.model, self.sched, tokens.data_ptr(), seq_lens.data_ptr(),
                    block_tables.data_ptr(), tokens.numel(), block_tables.shape[1],
                    k_pool.data_ptr(), v_pool.data_ptr(), k_pool.shape[1], self.ws_ptr,
                    self.ws_bytes, logits.data_ptr(), st)

    def check(self, stream=None) -> None:
        import torch
        st = (stream or torch.cuda.current_stream()).cuda_stream
        check_step(self.sched, self.ws_ptr, st)

    def region(self, name: str, dtype, count: int):
        """A view of a named workspace region (inspection)."""
        import torch
        off = self.sched.workspace_offset(name)
        if off < 0:
            raise KeyError(name)
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return self.workspace[self.ws_base + off:self.ws_base + off + nbytes].view(dtype)


def config_from(shape) -> MkConfig:
    """MkConfig from any object with the shape's attribute names."""
    return MkConfig(shape.n_layers, shape.hidden, shape.n_q, shape.n_kv, shape.head_dim,
                    shape.n_experts, shape.top_k, shape.inter, shape.vocab, shape.page_size,
                    shape.window, shape.full_period, shape.rope_base, shape.eps,
                    int(getattr(shape, "expert_fp8", False)), int(getattr(shape, "expert_fp4", False)))


def weights_from(tensors: dict) -> MkWeights:
    """MkWeights from a dict of device tensors named like the C struct fields."""
    def ptr(k):
        t = tensors.get(k)
        return t.data_ptr() if t is not None else None
    return MkWeights(*[ptr(n) for n, _ in MkWeights._fields_])
