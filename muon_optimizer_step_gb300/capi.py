"""ctypes binding of libmuon.so: the C entry points under the same names.

Only argument marshalling happens here (torch tensors -> device pointers, Python
lists -> host pointer arrays, a torch stream -> cudaStream_t); every step of the
optimizer runs in the library's CUDA kernels.  Importing this module loads the library
and raises if it has not been built: there is no other code path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# MUON_LIB may name another build of the library (e.g. libmuon_debug.so, whose kernels
# range-check every table entry they use); the default is the in-tree libmuon.so.
LIB_PATH = os.environ.get("MUON_LIB") or os.path.join(_HERE, "libmuon.so")

MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_ALIGNMENT = 2
MUON_ERR_CUDA = 3
MUON_ERR_TIMEOUT = 4
MUON_ERR_OOM = 5
MUON_ERR_UNSUPPORTED = 6
MUON_ERR_DEVICE_CHECK = 7
MUON_NS_BF16 = 0
MUON_NS_FP32 = 1
MUON_NS_SPLIT_FP32 = 2
MUON_MAX_SHARDS = 128
WORKSPACE_ALIGN = 1024

_STATUS_NAMES = {0: "MUON_OK", 1: "MUON_ERR_INVALID_ARG", 2: "MUON_ERR_ALIGNMENT",
                 3: "MUON_ERR_CUDA", 4: "MUON_ERR_TIMEOUT", 5: "MUON_ERR_OOM",
                 6: "MUON_ERR_UNSUPPORTED", 7: "MUON_ERR_DEVICE_CHECK"}

# (name, restype, argtypes) of every entry point declared in include/muon.h.
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_PP = ctypes.POINTER(ctypes.c_void_p)


class GroupHparams(ctypes.Structure):
    """muon_group_hparams: one optimizer group's hyper-parameters."""
    _fields_ = [("lr", ctypes.c_float), ("wd", ctypes.c_float), ("mu", ctypes.c_float),
                ("nesterov", ctypes.c_int32)]

SIGNATURES = [
    ("muon_abi_version", _I32, []),
    ("muon_last_error", ctypes.c_char_p, []),
    ("muon_layout_create", _I32, [ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_uint8), _I32,
                                  _I32, _I32, ctypes.POINTER(_P)]),
    ("muon_layout_destroy", _I32, [_P]),
    ("muon_layout_numel", _I32, [_P, ctypes.POINTER(_I64)]),
    ("muon_layout_shard_len", _I32, [_P, ctypes.POINTER(_I64)]),
    ("muon_layout_workspace_bytes", _I32, [_P, ctypes.POINTER(ctypes.c_size_t)]),
    ("muon_layout_full_numel", _I32, [_P, ctypes.POINTER(_I64)]),
    ("muon_full_offsets", _I32, [_P, ctypes.POINTER(_I64)]),
    ("muon_step", _I32, [_PP, _PP, _PP, _P, _P, _F, _F, _F, _I32, _I32, _P]),
    ("muon_compute_momentum_inputs", _I32, [_PP, _PP, _P, _P, _F, _I32, _P]),
    ("muon_orthogonalize_updates", _I32, [_P, _P, _I32, _P]),
    ("muon_apply_local_updates", _I32, [_PP, _P, _P, _F, _F, _I32, _P]),
    ("muon_orthogonalize_apply", _I32, [_PP, _P, _P, _F, _F, _I32, _P]),
    ("muon_layout_set_groups", _I32, [_P, ctypes.POINTER(_I32), _I32]),
    ("muon_step_grouped", _I32, [_PP, _PP, _PP, _P, _P, ctypes.POINTER(GroupHparams), _I32, _P]),
    ("muon_assign_owners", _I32, [_P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(ctypes.c_double)]),
    ("muon_exchange_plan", _I32, [_P, ctypes.POINTER(_I32), _I32, _P, ctypes.POINTER(_I64), _P,
                                  ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                  ctypes.POINTER(_I64)]),
    ("muon_gather_full", _I32, [_P, _PP, _P, _P]),
    ("muon_scatter_updates", _I32, [_P, _P, _PP, _P]),
    ("muon_orthogonalize_full", _I32, [_P, _P, _P, _P, _I32, _P]),
    ("muon_export_input", _I32, [_P, _P, _P, _P]),
    ("muon_export_update", _I32, [_P, _P, _I32, _P, _P]),
    ("muon_orthogonalize_full_noalloc", _I32, [_P, _P, _P, _I32, _P]),
    ("muon_check", _I32, [_P]),
    ("muon_selftest_wait_timeout", _I32, [_I64, _P]),
    ("muon_debug_build", _I32, []),
    ("muon_selftest_device_check", _I32, [_P]),
    ("muon_layout_ns_kernel", _I32, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32),
                                     ctypes.POINTER(_I32)]),
    ("muon_layout_fused_apply", _I32, [_P, ctypes.POINTER(_I32)]),
]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()'); this package has no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib.muon_last_error().decode(errors="replace")
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status: int, where: str):
    if status != MUON_OK:
        raise MuonError(status, where)


# ------------------------------------------------------------------ marshalling helpers
def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _shard_array(layout, shards, name):
    """A host array of n_shards device pointers from a tensor or a list of tensors."""
    if not isinstance(shards, (list, tuple)):
        shards = [shards]
    if len(shards) != layout.n_shards:
        raise ValueError(f"{name}: expected {layout.n_shards} shard(s), got {len(shards)}")
    for s in shards:
        if isinstance(s, int):
            continue
        import torch
        if s.dtype != torch.float32 or not s.is_contiguous() or s.device.type != "cuda":
            raise ValueError(f"{name}: shards must be contiguous float32 CUDA tensors")
        if s.numel() < layout.shard_len:
            raise ValueError(f"{name}: shard has {s.numel()} elements, layout needs {layout.shard_len}")
    arr = (ctypes.c_void_p * max(1, len(shards)))()
    for i, s in enumerate(shards):
        arr[i] = s if isinstance(s, int) else s.data_ptr()
    return arr


class Layout:
    """Owns a muon_layout handle (see muon_layout_create)."""

    def __init__(self, handle, shapes, is_matrix, n_shards, ns_dtype):
        self.handle = handle
        self.shapes = shapes
        self.is_matrix = is_matrix
        self.n_shards = n_shards
        self.ns_dtype = ns_dtype
        v = _I64()
        _check(lib.muon_layout_numel(handle, ctypes.byref(v)), "muon_layout_numel")
        self.numel = v.value
        _check(lib.muon_layout_shard_len(handle, ctypes.byref(v)), "muon_layout_shard_len")
        self.shard_len = v.value
        _check(lib.muon_layout_full_numel(handle, ctypes.byref(v)), "muon_layout_full_numel")
        self.full_numel = v.value
        b = ctypes.c_size_t()
        _check(lib.muon_layout_workspace_bytes(handle, ctypes.byref(b)),
               "muon_layout_workspace_bytes")
        self.workspace_bytes = b.value
        offs = (_I64 * max(1, len(shapes)))()
        _check(lib.muon_full_offsets(handle, offs), "muon_full_offsets")
        self.full_offsets = [offs[i] for i in range(len(shapes))]

    def close(self):
        if self.handle:
            lib.muon_layout_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def _as_parameter_(self):
        return self.handle


def muon_layout_create(shapes, n_shards=1, ns_dtype=MUON_NS_BF16, is_matrix=None) -> Layout:
    shapes = [(int(r), int(c)) for r, c in shapes]
    n = len(shapes)
    flat = (_I64 * max(1, 2 * n))(*[v for rc in shapes for v in rc])
    flags = None
    if is_matrix is not None:
        is_matrix = [1 if f else 0 for f in is_matrix]
        if len(is_matrix) != n:
            raise ValueError("is_matrix must have one flag per shape")
        flags = (ctypes.c_uint8 * max(1, n))(*is_matrix)
    if isinstance(ns_dtype, str):
        ns_dtype = {"bf16": MUON_NS_BF16, "fp32": MUON_NS_FP32, "split": MUON_NS_SPLIT_FP32}[ns_dtype]
    h = ctypes.c_void_p()
    _check(lib.muon_layout_create(flat, flags, n, int(n_shards), int(ns_dtype), ctypes.byref(h)),
           "muon_layout_create")
    return Layout(h, shapes, is_matrix, int(n_shards), int(ns_dtype))


def workspace_tensor(layout: Layout, device="cuda"):
    """A uint8 CUDA tensor of layout.workspace_bytes whose data_ptr is 1024-byte aligned."""
    import torch
    raw = torch.empty(layout.workspace_bytes + WORKSPACE_ALIGN, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % WORKSPACE_ALIGN
    ws = raw[off: off + layout.workspace_bytes]
    ws._muon_base = raw  # keep the allocation alive with the view
    return ws


def muon_step(flat_params, flat_grads, flat_momentum, layout, workspace, lr, wd, mu,
              nesterov=True, ns_steps=5, stream=None):
    _check(lib.muon_step(_shard_array(layout, flat_params, "flat_params"),
                         _shard_array(layout, flat_grads, "flat_grads"),
                         _shard_array(layout, flat_momentum, "flat_momentum"),
                         layout.handle, _ptr(workspace), float(lr), float(wd), float(mu),
                         1 if nesterov else 0, int(ns_steps), _stream_handle(stream)),
           "muon_step")


def muon_layout_set_groups(layout, group_of, n_groups):
    arr = (_I32 * max(1, len(group_of)))(*[int(g) for g in group_of])
    _check(lib.muon_layout_set_groups(layout.handle, arr, int(n_groups)), "muon_layout_set_groups")
    layout.n_groups = int(n_groups)


def muon_step_grouped(flat_params, flat_grads, flat_momentum, layout, workspace, groups,
                      ns_steps=5, stream=None):
    """groups: a sequence of (lr, wd, mu, nesterov), one per optimizer group."""
    arr = (GroupHparams * max(1, len(groups)))(
        *[GroupHparams(float(lr), float(wd), float(mu), 1 if nest else 0)
          for lr, wd, mu, nest in groups])
    _check(lib.muon_step_grouped(_shard_array(layout, flat_params, "flat_params"),
                                 _shard_array(layout, flat_grads, "flat_grads"),
                                 _shard_array(layout, flat_momentum, "flat_momentum"),
                                 layout.handle, _ptr(workspace), arr, int(ns_steps),
                                 _stream_handle(stream)), "muon_step_grouped")


def muon_compute_momentum_inputs(flat_grads, flat_momentum, layout, workspace, mu,
                                 nesterov=True, stream=None):
    _check(lib.muon_compute_momentum_inputs(
        _shard_array(layout, flat_grads, "flat_grads"),
        _shard_array(layout, flat_momentum, "flat_momentum"), layout.handle, _ptr(workspace),
        float(mu), 1 if nesterov else 0, _stream_handle(stream)), "muon_compute_momentum_inputs")


def muon_orthogonalize_updates(layout, workspace, ns_steps=5, stream=None):
    _check(lib.muon_orthogonalize_updates(layout.handle, _ptr(workspace), int(ns_steps),
                                          _stream_handle(stream)), "muon_orthogonalize_updates")


def muon_apply_local_updates(flat_params, layout, workspace, lr, wd, ns_steps=5, stream=None):
    _check(lib.muon_apply_local_updates(_shard_array(layout, flat_params, "flat_params"),
                                        layout.handle, _ptr(workspace), float(lr), float(wd),
                                        int(ns_steps), _stream_handle(stream)),
           "muon_apply_local_updates")


def muon_orthogonalize_apply(flat_params, layout, workspace, lr, wd, ns_steps=5, stream=None):
    _check(lib.muon_orthogonalize_apply(_shard_array(layout, flat_params, "flat_params"),
                                        layout.handle, _ptr(workspace), float(lr), float(wd),
                                        int(ns_steps), _stream_handle(stream)),
           "muon_orthogonalize_apply")


def muon_assign_owners(layout, ns_steps=5):
    """(owner per parameter, flop total per rank) for one rank per shard."""
    owner = (_I32 * max(1, len(layout.shapes)))()
    cost = (ctypes.c_double * max(1, layout.n_shards))()
    _check(lib.muon_assign_owners(layout.handle, int(ns_steps), owner, cost), "muon_assign_owners")
    return [owner[i] for i in range(len(layout.shapes))], [cost[s] for s in range(layout.n_shards)]


class Xfer(ctypes.Structure):
    """muon_xfer: one run of a matrix's flat elements moved between a shard and its
    owner's packed buffer."""
    _fields_ = [("param", ctypes.c_int32), ("src_rank", ctypes.c_int32),
                ("dst_rank", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("shard_off", ctypes.c_int64), ("owner_off", ctypes.c_int64),
                ("len", ctypes.c_int64)]


def muon_exchange_plan(layout, owner, rank):
    """(sends, recvs, owned_numel, owned_offsets) of the owner exchange for `rank`: sends
    and recvs are lists of dicts with the muon_xfer fields."""
    n = len(layout.shapes)
    own = (_I32 * max(1, n))(*[int(o) for o in owner])
    ns, nr, owned = _I64(0), _I64(0), _I64(0)
    _check(lib.muon_exchange_plan(layout.handle, own, int(rank), None, ctypes.byref(ns), None,
                                  ctypes.byref(nr), ctypes.byref(owned), None),
           "muon_exchange_plan")
    snd = (Xfer * max(1, ns.value))()
    rcv = (Xfer * max(1, nr.value))()
    offs = (_I64 * max(1, n))()
    _check(lib.muon_exchange_plan(layout.handle, own, int(rank), snd, ctypes.byref(ns), rcv,
                                  ctypes.byref(nr), ctypes.byref(owned), offs),
           "muon_exchange_plan")

    def rows(arr, k):
        return [{f: getattr(arr[i], f) for f, _ in Xfer._fields_ if f != "pad_"}
                for i in range(k)]
    return rows(snd, ns.value), rows(rcv, nr.value), owned.value, [offs[i] for i in range(n)]


def muon_gather_full(layout, shards, full, stream=None):
    _check(lib.muon_gather_full(layout.handle, _shard_array(layout, shards, "shards"), _ptr(full),
                                _stream_handle(stream)), "muon_gather_full")


def muon_scatter_updates(layout, full, shards, stream=None):
    _check(lib.muon_scatter_updates(layout.handle, _ptr(full), _shard_array(layout, shards, "shards"),
                                    _stream_handle(stream)), "muon_scatter_updates")


def muon_orthogonalize_full(layout, workspace, full_in, full_out, ns_steps=5, stream=None):
    _check(lib.muon_orthogonalize_full(layout.handle, _ptr(workspace), _ptr(full_in),
                                       _ptr(full_out), int(ns_steps), _stream_handle(stream)),
           "muon_orthogonalize_full")


def muon_orthogonalize_full_noalloc(layout, full_in, full_out, ns_steps=5, stream=None):
    """Like muon_orthogonalize_full, but with no workspace argument and no device
    allocation: for callers that cannot allocate device memory where they orthogonalize
    (fp32 layouts up to 32 MiB of tables plus workspace; see include/muon.h)."""
    _check(lib.muon_orthogonalize_full_noalloc(layout.handle, _ptr(full_in), _ptr(full_out),
                                               int(ns_steps), _stream_handle(stream)),
           "muon_orthogonalize_full_noalloc")


def muon_export_input(layout, workspace, full_out, stream=None):
    _check(lib.muon_export_input(layout.handle, _ptr(workspace), _ptr(full_out),
                                 _stream_handle(stream)), "muon_export_input")


def muon_export_update(layout, workspace, ns_steps, full_out, stream=None):
    _check(lib.muon_export_update(layout.handle, _ptr(workspace), int(ns_steps), _ptr(full_out),
                                  _stream_handle(stream)), "muon_export_update")


def muon_check(stream=None):
    _check(lib.muon_check(_stream_handle(stream)), "muon_check")


def muon_check_status(stream=None) -> int:
    """Like muon_check but returns the status instead of raising."""
    return lib.muon_check(_stream_handle(stream))


def muon_selftest_wait_timeout(budget_cycles, stream=None):
    _check(lib.muon_selftest_wait_timeout(int(budget_cycles), _stream_handle(stream)),
           "muon_selftest_wait_timeout")


def muon_debug_build() -> bool:
    """Whether the loaded library was built with device-side range checks."""
    return bool(lib.muon_debug_build())


def muon_selftest_device_check(stream=None):
    _check(lib.muon_selftest_device_check(_stream_handle(stream)), "muon_selftest_device_check")


def muon_layout_ns_kernel(layout) -> dict:
    """The Newton-Schulz kernel `layout` runs on the current device:
    {"tile_shape": 1 single CTA | 2 CTA pair | 3 CTA pair with 256x512 tiles (0: none),
     "units": int, "persistent": bool}."""
    shape, units, pers = _I32(), _I32(), _I32()
    _check(lib.muon_layout_ns_kernel(layout.handle, ctypes.byref(shape), ctypes.byref(units),
                                     ctypes.byref(pers)), "muon_layout_ns_kernel")
    return {"tile_shape": int(shape.value), "units": int(units.value),
            "persistent": bool(pers.value)}


def muon_layout_fused_apply(layout) -> bool:
    """True when muon_step / muon_orthogonalize_apply apply the update to W inside the last
    Newton-Schulz Update on the current device, False when a separate apply pass runs."""
    f = _I32()
    _check(lib.muon_layout_fused_apply(layout.handle, ctypes.byref(f)), "muon_layout_fused_apply")
    return bool(f.value)


def muon_last_error() -> str:
    return lib.muon_last_error().decode(errors="replace")


def muon_abi_version() -> int:
    return lib.muon_abi_version()
