"""Thin Python binding of libpw.so, the fused mixed-precision APL MoE layer
for GB300 (sm_103a).

The functions keep the C ABI's names (pw_pack, pw_set_commit, pw_reload_async,
pw_moe_forward, ...) and only marshal arguments: torch tensors become raw
pointers, the current torch stream becomes the CUDA stream.  Every step of the
layer runs in the library's own kernels; there is no fallback path, and every
entry point raises if the library has not been built.

PyTorch supplies device memory (plane pages, tables, descriptors, workspace)
and streams; the library allocates none of its own.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpw.so")
CHECK_LIB_PATH = os.path.join(HERE, "libpw_check.so")

PW_OK = 0
PW_EINVAL = -1
PW_ECUDA = -2
PW_ENOTRESIDENT = -3
PW_ERELOAD = -4
PW_ETIMEOUT = -5
PW_ENOMEM = -6
PW_EDEVICE = -7
PW_STATUS_NAN_LOGIT = 1
PW_STATUS_TIMEOUT = 2
PW_STATUS_BAD_DESC = 4
PW_STATUS_BOUNDS = 8
PW_WS_H, PW_WS_Y = 0, 1
PW_PLANE_HOST, PW_PLANE_HOST_PAGED, PW_PLANE_MOVING, PW_PLANE_DEVICE = 0, 1, 2, 3
KIND_GATE_UP = 0
KIND_DOWN = 1
MAX_BITS = 8

_lib = None

_sz = ctypes.c_size_t
_vp = ctypes.c_void_p
_i = ctypes.c_int
_pi = ctypes.POINTER(ctypes.c_int)

_SIGS = {
    "pw_last_error": (ctypes.c_char_p, []),
    "pw_plane_bytes": (_sz, [_i, _i]),
    "pw_lut_bytes": (_sz, [_i, _i, _i]),
    "pw_lut_offset": (_sz, [_i, _i, _i]),
    "pw_pack": (_i, [_vp, _i, _i, _i, _vp, _i, _vp, _vp]),
    "pw_tile_planes": (_i, [_vp, _i, _i, _i, _vp]),
    "pw_desc_bytes": (_sz, [_i, _i]),
    "pw_table_create": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _i, _vp, _sz, _vp]),
    "pw_block_register": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, ctypes.POINTER(_vp), _vp, _i, _vp]),
    "pw_set_commit": (_i, [_vp, _i, _i, _i, _i, _vp]),
    "pw_reload_async": (_i, [_vp, _i, _i, _i, _i, _vp]),
    "pw_reload_query": (_i, [_vp, _i, _i, _i]),
    "pw_reload_many": (_i, [_vp, _i, _pi, _pi, _pi, _pi, _vp, _pi]),
    "pw_set_commit_many": (_i, [_vp, _i, _pi, _pi, _pi, _pi, _vp]),
    "pw_mover_start": (_i, [_vp, _vp, _sz]),
    "pw_mover_submit": (_i, [_vp, _i, _pi, _pi, _pi, _pi]),
    "pw_commit_arrived": (_i, [_vp, _vp, _pi, _pi]),
    "pw_block_state": (_i, [_vp, _i, _i, _i, _pi, _pi, _pi]),
    "pw_table_destroy": (_i, [_vp]),
    "pw_debug_fail_next_reload": (_i, [_vp]),
    "pw_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "pw_workspace_offset": (_sz, [_i, _i, _i, _i, _i, _i]),
    "pw_moe_forward": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "pw_moe_forward_host": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "pw_workspace_status": (_i, [_vp, _vp, _pi]),
    "pw_moe_forward_noalloc": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp]),
    "pw_noalloc_status": (_i, [_vp, _pi]),
    "pw_profile_attach": (_i, [ctypes.POINTER(_vp), _i]),
    "pw_stats_attach": (_i, [_vp, _vp, ctypes.c_float]),
    "pw_plan_bits": (_i, [_i, _vp, _vp, _vp, _vp, _vp, _i, ctypes.c_double, _i, _i, _i, ctypes.c_double,
                          _vp, ctypes.POINTER(ctypes.c_int64)]),
    "pw_plan_apply": (_i, [_vp, _vp, _vp, _pi, _pi]),
    "pw_block_release": (_i, [_vp, _i, _i, _i, _i, ctypes.POINTER(_vp)]),
    "pw_block_attach_pages": (_i, [_vp, _i, _i, _i, ctypes.POINTER(_vp)]),
    "pw_plane_states": (_i, [_vp, _i, _i, _i, _pi]),
}


class PWError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (status {code})")
        self.code = code


def lib():
    """Loads libpw.so (once).  Raises if it has not been built.  With the
    environment variable PW_CHECK=1, loads libpw_check.so instead: the same
    library with device-side bounds checks that set PW_STATUS_BOUNDS."""
    global _lib
    if _lib is None:
        path = CHECK_LIB_PATH if os.environ.get("PW_CHECK") == "1" else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first "
                               "(python -m any_precision_weight_gb300.build)")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return sorted(_SIGS)


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise PWError(rc, f"{what}: {lib().pw_last_error().decode()}")
    return rc


def _ptr(t):
    """Address of a torch tensor or numpy array (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


# ----------------------------------------------------------------------------- format

def pw_plane_bytes(R: int, K: int) -> int:
    return lib().pw_plane_bytes(R, K)


def pw_lut_bytes(R: int, b_min: int, n_bits: int) -> int:
    return lib().pw_lut_bytes(R, b_min, n_bits)


def pw_lut_offset(R: int, b_min: int, b: int) -> int:
    return lib().pw_lut_offset(R, b_min, b)


def pw_pack(idx: np.ndarray, parent_lut: np.ndarray, n_bits: int = 8, b_min: int = 3,
            planes_out=None, luts_out=None):
    """Packs uint8 parent indices [R][K] and the fp16 parent table [R][2^n].

    Returns (planes uint32 [n][R][K/32], luts uint16 flat) as numpy arrays, or
    fills the given host buffers (numpy arrays over any host memory).
    """
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    par = np.ascontiguousarray(parent_lut, dtype=np.float16).view(np.uint16)
    R, K = idx.shape
    if planes_out is None:
        planes_out = np.empty((n_bits, R, K // 32), dtype=np.uint32)
    if luts_out is None:
        luts_out = np.empty(pw_lut_bytes(R, b_min, n_bits) // 2, dtype=np.uint16)
    _check(lib().pw_pack(_ptr(idx), R, K, n_bits, _ptr(par), b_min, _ptr(planes_out),
                         _ptr(luts_out)), "pw_pack")
    return planes_out, luts_out


def pw_tile_planes(planes: np.ndarray, out=None):
    """Reorders pw_pack planes uint32 [n][R][K/32] into the device page layout
    (returned as a flat uint32 array of the same size, or written into ``out``)."""
    planes = np.ascontiguousarray(planes, dtype=np.uint32)
    n, R, W = planes.shape
    if out is None:
        out = np.empty(planes.size, dtype=np.uint32)
    _check(lib().pw_tile_planes(_ptr(planes), n, R, W * 32, _ptr(out)), "pw_tile_planes")
    return out


def pw_profile_attach(events):
    """Next pw_moe_forward on this thread records these 5 torch.cuda.Events at its
    kernel boundaries (before routing, after routing, gate_up, down, combine);
    None entries are not recorded.  The decode path is one kernel: it records
    events[0] before it and events[1..4] after it."""
    if not events:
        return lib().pw_profile_attach(None, 0)
    arr = (_vp * len(events))(*[e.cuda_event if e is not None else None for e in events])
    return _check(lib().pw_profile_attach(arr, len(events)), "pw_profile_attach")


# ----------------------------------------------------------------------------- page table

def pw_plan_bits(R, K, sens, mass, n_experts, hot_mass, hot_floor, target_bytes, resid=None,
                 b_min: int = 3, n_bits: int = MAX_BITS):
    """The native planner on host arrays (one entry per block).  Returns
    (bits int32 array, resident bytes of the plan)."""
    R = np.ascontiguousarray(R, dtype=np.int32)
    K = np.ascontiguousarray(K, dtype=np.int32)
    sens = np.ascontiguousarray(sens, dtype=np.float64)
    mass = np.ascontiguousarray(mass, dtype=np.float64)
    rs = None if resid is None else np.ascontiguousarray(resid, dtype=np.float64)
    out = np.empty(len(R), dtype=np.int32)
    res = ctypes.c_int64()
    _check(lib().pw_plan_bits(len(R), _ptr(R), _ptr(K), _ptr(sens), _ptr(rs), _ptr(mass), int(n_experts),
                              float(hot_mass), int(hot_floor), int(b_min), int(n_bits), float(target_bytes),
                              _ptr(out), ctypes.byref(res)), "pw_plan_bits")
    return out, res.value


class PagedMoE:
    """Owns the device memory of one model's MoE blocks and the C page table.

    Plane pages, tables and descriptors are torch CUDA tensors; host backing
    copies are pinned torch CPU tensors.  Only the pages a block may use
    (``alloc_planes``) are allocated on the device.
    """

    def __init__(self, n_layers: int, n_experts: int, H: int, I: int, device="cuda", stream=None,
                 guard: int = 0):
        """guard > 0: every device buffer this object allocates (descriptors,
        plane pages, tables, workspaces) gets canary regions of that many bytes
        on both sides (``guard.GuardSet``), checked by ``corrupted_guards``."""
        import torch
        from .guard import GuardSet
        self.L, self.E, self.H, self.I = n_layers, n_experts, H, I
        self.device = torch.device(device)
        self.guards = GuardSet(guard) if guard > 0 else None
        nb = lib().pw_desc_bytes(n_layers, n_experts)
        self._desc = self._alloc(nb + 128, "descriptors")
        self._desc.zero_()
        base = self._desc.data_ptr()
        self._desc_ptr = base + ((-base) % 128)
        h = _vp()
        _check(lib().pw_table_create(ctypes.byref(h), n_layers, n_experts, H, I, self._desc_ptr, nb,
                                     _stream(stream)), "pw_table_create")
        self._t = h
        self._keep = {}

    def _alloc(self, nbytes: int, name: str):
        import torch
        if self.guards is None:
            return torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.guards.alloc(nbytes, self.device, name)

    def corrupted_guards(self) -> list:
        """Guard regions changed since allocation: [(buffer, side, offset)]."""
        return [] if self.guards is None else self.guards.corrupted()

    def rows_cols(self, kind: int):
        return (2 * self.I, self.H) if kind == KIND_GATE_UP else (self.H, self.I)

    def register(self, layer: int, expert: int, kind: int, planes_host, luts_host, q_init: int,
                 n_bits: int = 8, b_min: int = 3, alloc_planes: int | None = None, stream=None,
                 per_plane: bool = False):
        """planes_host / luts_host: pinned torch CPU tensors (or numpy arrays) in
        pw_pack layout; kept alive by this object.  per_plane: one device
        tensor per plane (so released planes free their memory) instead of one
        tensor for all of the block's pages."""
        import torch
        R, K = self.rows_cols(kind)
        pb = pw_plane_bytes(R, K)
        na = n_bits if alloc_planes is None else max(q_init, min(alloc_planes, n_bits))
        tag = f"{layer}/{expert}/{kind}"
        luts = self._alloc(pw_lut_bytes(R, b_min, n_bits), f"tables {tag}")
        if per_plane:
            pages = [self._alloc(pb, f"plane {p} {tag}") if p < na else None for p in range(n_bits)]
            ptrs = (_vp * n_bits)(*[pg.data_ptr() if pg is not None else None for pg in pages])
        else:
            pages = self._alloc(na * pb, f"planes {tag}")
            ptrs = (_vp * n_bits)(*[pages.data_ptr() + p * pb if p < na else None for p in range(n_bits)])
        _check(lib().pw_block_register(self._t, layer, expert, kind, n_bits, b_min, _ptr(planes_host),
                                       _ptr(luts_host), ptrs, luts.data_ptr(), q_init, _stream(stream)),
               "pw_block_register")
        self._keep[(layer, expert, kind)] = (pages, luts, planes_host, luts_host)

    def pages(self, layer, expert, kind):
        """(device plane pages tensor, device table tensor) of one block."""
        return self._keep[(layer, expert, kind)][:2]

    def device_bytes(self) -> int:
        def nb(pages):
            if isinstance(pages, list):
                return sum(p.numel() for p in pages if p is not None)
            return pages.numel()
        return sum(nb(v[0]) + v[1].numel() for v in self._keep.values())

    def pw_block_release(self, layer, expert, kind, keep, stream=None):
        """Offloads planes [keep, n) of a block.  Per-plane blocks drop their
        page tensors once the stream has passed every earlier forward.
        Returns the released device addresses (None where none)."""
        import torch
        out = (_vp * MAX_BITS)()
        _check(lib().pw_block_release(self._t, layer, expert, kind, keep, out), "pw_block_release")
        rel = [out[p] for p in range(MAX_BITS)]
        pages = self._keep[(layer, expert, kind)][0]
        if isinstance(pages, list) and any(rel):
            (stream or torch.cuda.current_stream()).synchronize()
            for p in range(MAX_BITS):
                if rel[p] and p < len(pages):
                    pages[p] = None
        return rel

    def pw_block_attach_pages(self, layer, expert, kind):
        """Gives a per-plane block fresh device pages for every plane without one."""
        import torch
        pages = self._keep[(layer, expert, kind)][0]
        assert isinstance(pages, list), "attach_pages needs a block registered with per_plane=True"
        R, K = self.rows_cols(kind)
        pb = pw_plane_bytes(R, K)
        new = [None] * MAX_BITS
        for p in range(len(pages)):
            if pages[p] is None:
                new[p] = self._alloc(pb, f"plane {p} {layer}/{expert}/{kind} (attached)")
        ptrs = (_vp * MAX_BITS)(*[t.data_ptr() if t is not None else None for t in new])
        _check(lib().pw_block_attach_pages(self._t, layer, expert, kind, ptrs), "pw_block_attach_pages")
        for p in range(len(pages)):
            if new[p] is not None:
                pages[p] = new[p]

    def pw_plane_states(self, layer, expert, kind):
        st = (_i * MAX_BITS)()
        _check(lib().pw_plane_states(self._t, layer, expert, kind, st), "pw_plane_states")
        return [st[p] for p in range(MAX_BITS)]

    def pw_set_commit(self, layer, expert, kind, q, stream=None):
        return _check(lib().pw_set_commit(self._t, layer, expert, kind, q, _stream(stream)),
                      "pw_set_commit")

    def pw_reload_async(self, layer, expert, kind, q_target, stream=None):
        return _check(lib().pw_reload_async(self._t, layer, expert, kind, q_target, _stream(stream)),
                      "pw_reload_async")

    @staticmethod
    def _columns(items):
        """[(layer, expert, kind, q), ...] -> four ctypes int arrays."""
        n = len(items)
        cols = [(ctypes.c_int * n)(*[int(it[j]) for it in items]) for j in range(4)]
        return n, cols

    def pw_reload_many(self, items, stream=None):
        """items: [(layer, expert, kind, q_target)].  Returns the number enqueued;
        raises PWError on the first failing block."""
        n, (l, e, k, q) = self._columns(items)
        done = _i()
        rc = lib().pw_reload_many(self._t, n, l, e, k, q, _stream(stream), ctypes.byref(done))
        _check(rc, "pw_reload_many")
        return done.value

    def pw_set_commit_many(self, items, stream=None):
        """items: [(layer, expert, kind, q)], committed at one stream boundary."""
        n, (l, e, k, q) = self._columns(items)
        return _check(lib().pw_set_commit_many(self._t, n, l, e, k, q, _stream(stream)),
                      "pw_set_commit_many")

    def pw_mover_start(self, stream, max_inflight_bytes: int = 64 << 20):
        """Starts the table's reload mover thread on the given copy stream."""
        return _check(lib().pw_mover_start(self._t, _stream(stream), max_inflight_bytes),
                      "pw_mover_start")

    def pw_mover_submit(self, items):
        """items: [(layer, expert, kind, q_target)], reloaded in order and
        committed by pw_commit_arrived once landed."""
        n, (l, e, k, q) = self._columns(items)
        return _check(lib().pw_mover_submit(self._t, n, l, e, k, q), "pw_mover_submit")

    def pw_commit_arrived(self, stream=None):
        """Commits every landed mover reload; returns (committed, outstanding)."""
        c, o = _i(), _i()
        _check(lib().pw_commit_arrived(self._t, _stream(stream), ctypes.byref(c), ctypes.byref(o)),
               "pw_commit_arrived")
        return c.value, o.value

    def pw_stats_attach(self, stats=None, alpha: float = 0.05):
        """Attaches a float32 CUDA tensor [L][E] of routing-mass moving averages
        (updated by every forward), or detaches with None."""
        if stats is not None:
            import torch
            assert stats.dtype == torch.float32 and stats.is_contiguous()
            assert stats.numel() == self.L * self.E
        self._stats = stats
        return _check(lib().pw_stats_attach(self._t, _ptr(stats), float(alpha)), "pw_stats_attach")

    def pw_plan_apply(self, desired, stream=None):
        """desired: int array [L][E][2] (0 = leave alone).  Returns (committed now,
        handed to the mover)."""
        d = np.ascontiguousarray(desired, dtype=np.int32).reshape(-1)
        assert d.size == self.L * self.E * 2
        a, b = _i(), _i()
        _check(lib().pw_plan_apply(self._t, _ptr(d), _stream(stream), ctypes.byref(a), ctypes.byref(b)),
               "pw_plan_apply")
        return a.value, b.value

    def pw_reload_query(self, layer, expert, kind) -> int:
        return _check(lib().pw_reload_query(self._t, layer, expert, kind), "pw_reload_query")

    def pw_block_state(self, layer, expert, kind):
        q, res, tgt = _i(), _i(), _i()
        _check(lib().pw_block_state(self._t, layer, expert, kind, ctypes.byref(q), ctypes.byref(res),
                                    ctypes.byref(tgt)), "pw_block_state")
        return q.value, res.value, tgt.value

    def pw_debug_fail_next_reload(self):
        return _check(lib().pw_debug_fail_next_reload(self._t), "pw_debug_fail_next_reload")

    def workspace_h(self, ws, T: int, top_k: int):
        """h (fp16 [T*top_k][I], permuted pair order) left in `ws` by the last forward."""
        import torch
        off = lib().pw_workspace_offset(T, self.E, top_k, self.H, self.I, PW_WS_H)
        n = T * top_k * self.I * 2
        return ws[off:off + n].view(torch.float16).view(T * top_k, self.I)

    def workspace_y(self, ws, T: int, top_k: int):
        """y (fp32 [T*top_k][H], permuted pair order) left in `ws` by the last forward."""
        import torch
        off = lib().pw_workspace_offset(T, self.E, top_k, self.H, self.I, PW_WS_Y)
        n = T * top_k * self.H * 4
        return ws[off:off + n].view(torch.float32).view(T * top_k, self.H)

    def workspace(self, T: int, top_k: int):
        nb = lib().pw_workspace_bytes(T, self.E, top_k, self.H, self.I)
        return self._alloc(max(nb, 256), f"workspace T={T}")

    def pw_moe_forward(self, layer, x, logits, top_k, renorm, residual=None, out=None, ws=None,
                       routing=False, stream=None):
        """x [T][H] fp16 and logits [T][E] fp32 CUDA tensors.  Returns out, or
        (out, topk_idx, topk_w, offsets, perm) with routing=True."""
        import torch
        T = x.shape[0]
        assert x.dtype == torch.float16 and logits.dtype == torch.float32
        assert x.is_contiguous() and logits.is_contiguous()
        if out is None:
            out = torch.empty_like(x)
        if ws is None:
            ws = self.workspace(T, top_k)
        ri = rw = ro = rp = None
        if routing:
            ri = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
            rw = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
            ro = torch.empty((self.E + 1,), dtype=torch.int32, device=x.device)
            rp = torch.empty((T * top_k,), dtype=torch.int32, device=x.device)
        _check(lib().pw_moe_forward(self._t, layer, _ptr(x), _ptr(logits), T, top_k, int(renorm),
                                    _ptr(residual), _ptr(out), _ptr(ri), _ptr(rw), _ptr(ro), _ptr(rp),
                                    _ptr(ws), ws.numel(), _stream(stream)), "pw_moe_forward")
        return (out, ri, rw, ro, rp) if routing else out

    def pw_moe_forward_host(self, layer, x_host, logits_host, top_k, renorm, out_host,
                            residual_host=None, ws=None, stream=None):
        """Host (pinned) inputs and output; synchronises the stream."""
        T = x_host.shape[0]
        if ws is None:
            ws = self.workspace(T, top_k)
        _check(lib().pw_moe_forward_host(self._t, layer, _ptr(x_host), _ptr(logits_host), T, top_k,
                                         int(renorm), _ptr(residual_host), _ptr(out_host), _ptr(ws),
                                         ws.numel(), _stream(stream)), "pw_moe_forward_host")
        return out_host

    def pw_moe_forward_noalloc(self, layer, x, logits, top_k, renorm, residual=None, out=None,
                               stream=None):
        """pw_moe_forward without a caller workspace: the library's fixed 8 MiB
        device scratch is used instead (for callers that cannot allocate).
        Calls that overlap on the GPU race on that scratch."""
        import torch
        assert x.dtype == torch.float16 and logits.dtype == torch.float32
        if out is None:
            out = torch.empty_like(x)
        _check(lib().pw_moe_forward_noalloc(self._t, layer, _ptr(x), _ptr(logits), x.shape[0], top_k,
                                            int(renorm), _ptr(residual), _ptr(out), _stream(stream)),
               "pw_moe_forward_noalloc")
        return out

    @staticmethod
    def workspace_status(ws, stream=None) -> int:
        st = _i()
        _check(lib().pw_workspace_status(_ptr(ws), _stream(stream), ctypes.byref(st)),
               "pw_workspace_status")
        return st.value

    @staticmethod
    def noalloc_status(stream=None) -> int:
        """Status bits of the last pw_moe_forward_noalloc ordered before `stream`'s work."""
        st = _i()
        _check(lib().pw_noalloc_status(_stream(stream), ctypes.byref(st)), "pw_noalloc_status")
        return st.value

    def close(self):
        if getattr(self, "_t", None):
            lib().pw_table_destroy(self._t)
            self._t = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
