"""Python binding of libspecverify (argument marshalling only).

Every function here forwards to the C ABI declared in ``include/specverify.h``; all of the verify step
runs in the library's CUDA kernels. PyTorch supplies device memory and streams. If the compiled library
is missing this module raises at import time: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_CUDA, SV_ERR_BAD_TOKEN, SV_ERR_BAD_OFFSETS = 0, 1, 2, 3, 4
SV_ERR_NONFINITE, SV_ERR_EMPTY_ROW, SV_ERR_TIMEOUT, SV_ERR_WORKSPACE, SV_ERR_CAPACITY = 5, 6, 7, 8, 9
SV_F32, SV_BF16 = 0, 1
SV_MAX_GAMMA = 31

# every exported symbol of the C ABI, in header order
EXPORTS = ("spec_verify", "spec_verify_workspace_size", "spec_verify_ex", "spec_verify_range", "spec_verify_noalloc",
           "spec_verify_commit", "spec_verify_fused", "spec_draft_ngram", "spec_verify_tree",
           "spec_shard_stats", "spec_shard_decide", "spec_shard_chunks", "spec_shard_sums", "spec_shard_finish",
           "spec_verify_status_from_bits", "spec_verify_status_string", "spec_verify_host")


class SvDebug(ctypes.Structure):
    _fields_ = [("row_lse", ctypes.c_void_p), ("row_argmax", ctypes.c_void_p),
                ("p_x", ctypes.c_void_p), ("q_x", ctypes.c_void_p), ("seq_mass", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("spin_limit", ctypes.c_uint32), ("order", ctypes.c_uint32),
                ("cluster", ctypes.c_uint32)]


class SvDeviceBuffers(ctypes.Structure):
    """Device staging buffers of spec_verify_host (device addresses)."""
    _fields_ = [("target_logits", ctypes.c_void_p), ("draft_logits", ctypes.c_void_p),
                ("draft_tokens", ctypes.c_void_p), ("seq_offsets", ctypes.c_void_p), ("gammas", ctypes.c_void_p),
                ("out_tokens", ctypes.c_void_p), ("out_num_accepted", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libspecverify.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    L.spec_verify.argtypes = [vp, vp, vp, vp, vp, i32, i32, f32, u64, u64, vp, vp]
    L.spec_verify.restype = ctypes.c_int
    L.spec_verify_workspace_size.argtypes = [i32, i32, i32]
    L.spec_verify_workspace_size.restype = sz
    L.spec_verify_ex.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp,
                                 vp, vp, sz, ctypes.POINTER(SvDebug), vp]
    L.spec_verify_ex.restype = ctypes.c_int
    L.spec_verify_range.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, f32, u64, u64, ctypes.c_uint32,
                                    vp, vp, vp, vp, sz, ctypes.POINTER(SvDebug), vp]
    L.spec_verify_range.restype = ctypes.c_int
    L.spec_verify_noalloc.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp,
                                      vp, ctypes.POINTER(SvDebug), vp]
    L.spec_verify_noalloc.restype = ctypes.c_int
    L.spec_verify_commit.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, vp, vp]
    L.spec_verify_commit.restype = ctypes.c_int
    L.spec_verify_fused.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp, vp, sz,
                                    vp, i32, vp, vp, vp]
    L.spec_verify_fused.restype = ctypes.c_int
    L.spec_draft_ngram.argtypes = [vp, i32, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    L.spec_draft_ngram.restype = ctypes.c_int
    L.spec_verify_tree.argtypes = [vp, ctypes.c_int, vp, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp, vp, vp,
                                   sz, vp]
    L.spec_verify_tree.restype = ctypes.c_int
    L.spec_verify_host.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp,
                                   ctypes.POINTER(SvDeviceBuffers), vp, vp, sz, vp]
    L.spec_verify_host.restype = ctypes.c_int
    L.spec_shard_stats.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp]
    L.spec_shard_stats.restype = ctypes.c_int
    L.spec_shard_decide.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, f32, i32, u64, u64, vp, vp, vp, vp, vp]
    L.spec_shard_decide.restype = ctypes.c_int
    L.spec_shard_chunks.argtypes = [i32, vp]
    L.spec_shard_chunks.restype = i32
    L.spec_shard_sums.argtypes = [i32, i32, vp, vp, vp, ctypes.c_int, vp, vp, i32, i32, f32, vp, vp]
    L.spec_shard_sums.restype = ctypes.c_int
    L.spec_shard_finish.argtypes = [i32, i32, vp, vp, vp, ctypes.c_int, vp, vp, vp, i32, i32, f32, vp, vp]
    L.spec_shard_finish.restype = ctypes.c_int
    L.spec_verify_status_from_bits.argtypes = [ctypes.c_uint32]
    L.spec_verify_status_from_bits.restype = ctypes.c_int
    L.spec_verify_status_string.argtypes = [ctypes.c_int]
    L.spec_verify_status_string.restype = ctypes.c_char_p
    return L


lib = _load()


def spec_verify(target_logits, draft_logits, draft_tokens, seq_offsets, gammas, B, V, temperature,
                seed, step, out_tokens, out_num_accepted) -> int:
    """Blocking bf16 form on the legacy default stream. Pointer arguments are device addresses (int)."""
    return lib.spec_verify(target_logits, draft_logits, draft_tokens, seq_offsets, gammas, B, V,
                           float(temperature), seed, step, out_tokens, out_num_accepted)


def spec_verify_workspace_size(B, V, max_gamma) -> int:
    return lib.spec_verify_workspace_size(B, V, max_gamma)


def spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                   temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                   workspace_bytes, debug: SvDebug | None, cuda_stream) -> int:
    """Asynchronous form. Pointer arguments are device addresses (int or None)."""
    return lib.spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                              max_gamma, float(temperature), seed, step, out_tokens, out_num_accepted,
                              device_status, workspace, workspace_bytes,
                              ctypes.byref(debug) if debug is not None else None, cuda_stream)


def spec_verify_range(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                      temperature, seed, step, seq_base, out_tokens, out_num_accepted, device_status, workspace,
                      workspace_bytes, debug: SvDebug | None, cuda_stream) -> int:
    """spec_verify_ex on a contiguous range of a larger batch whose sequence 0 is the batch's seq_base."""
    return lib.spec_verify_range(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                                 max_gamma, float(temperature), seed, step, seq_base, out_tokens, out_num_accepted,
                                 device_status, workspace, workspace_bytes,
                                 ctypes.byref(debug) if debug is not None else None, cuda_stream)


def spec_verify_noalloc(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                        temperature, seed, step, out_tokens, out_num_accepted, device_status,
                        debug: SvDebug | None, cuda_stream) -> int:
    """Allocation-free form for callers that cannot allocate device memory: the library's fixed 8 MiB
    scratch replaces the workspace. Calls sharing it must not overlap on the GPU."""
    return lib.spec_verify_noalloc(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                                   max_gamma, float(temperature), seed, step, out_tokens, out_num_accepted,
                                   device_status, ctypes.byref(debug) if debug is not None else None,
                                   cuda_stream)


def spec_verify_commit(out_tokens, out_num_accepted, seq_offsets, B, history, capacity, lengths, next_tokens,
                       device_status, cuda_stream) -> int:
    """Post-verify update on the device. Pointer arguments are device addresses (int or None)."""
    return lib.spec_verify_commit(out_tokens, out_num_accepted, seq_offsets, B, history, capacity, lengths,
                                  next_tokens, device_status, cuda_stream)


def spec_verify_fused(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                      temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                      workspace_bytes, history, capacity, lengths, next_tokens, cuda_stream) -> int:
    """Verify step with the post-verify update fused in. Pointer arguments are device addresses."""
    return lib.spec_verify_fused(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                                 max_gamma, float(temperature), seed, step, out_tokens, out_num_accepted,
                                 device_status, workspace, workspace_bytes, history, capacity, lengths,
                                 next_tokens, cuda_stream)


def spec_draft_ngram(history, capacity, lengths, B, n_min, n_max, gamma_max, draft_tokens, gammas, seq_offsets,
                     match_pos, device_status, cuda_stream) -> int:
    """N-gram drafts from the device-side histories. Pointer arguments are device addresses."""
    return lib.spec_draft_ngram(history, capacity, lengths, B, n_min, n_max, gamma_max, draft_tokens, gammas,
                                seq_offsets, match_pos, device_status, cuda_stream)


def spec_verify_tree(target_logits, dtype, draft_tokens, parents, seq_offsets, gammas, B, V, max_gamma, temperature,
                     seed, step, out_tokens, out_num_accepted, out_path, device_status, workspace, workspace_bytes,
                     cuda_stream) -> int:
    """Token-tree verification with point-mass candidates. Pointer arguments are device addresses."""
    return lib.spec_verify_tree(target_logits, dtype, draft_tokens, parents, seq_offsets, gammas, B, V, max_gamma,
                                float(temperature), seed, step, out_tokens, out_num_accepted, out_path, device_status,
                                workspace, workspace_bytes, cuda_stream)


def spec_verify_host(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                     temperature, seed, step, out_tokens, out_num_accepted, dev: SvDeviceBuffers | None,
                     device_status, workspace, workspace_bytes, cuda_stream) -> int:
    """Host-buffer form: host addresses for the inputs and outputs, device staging buffers in ``dev``."""
    return lib.spec_verify_host(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                                max_gamma, float(temperature), seed, step, out_tokens, out_num_accepted,
                                ctypes.byref(dev) if dev is not None else None, device_status, workspace,
                                workspace_bytes, cuda_stream)


def spec_shard_stats(shard_target, shard_draft, dtype, draft_tokens, seq_offsets, gammas, B, V, v0, Vs, max_gamma,
                     temperature, partials, device_status, cuda_stream) -> int:
    """Per-row statistics of one vocabulary shard's slice. Pointer arguments are device addresses."""
    return lib.spec_shard_stats(shard_target, shard_draft, dtype, draft_tokens, seq_offsets, gammas, B, V, v0, Vs,
                                max_gamma, float(temperature), partials, device_status, cuda_stream)


def spec_shard_decide(all_partials, S, bounds, draft_tokens, seq_offsets, gammas, B, V, max_gamma, temperature,
                      point_mass, seed, step, out_tokens, out_num_accepted, draws, device_status, cuda_stream) -> int:
    """Decisions from the gathered partials; `bounds` is a host sequence of S + 1 columns."""
    hb = (ctypes.c_int32 * (S + 1))(*[int(v) for v in bounds])
    return lib.spec_shard_decide(all_partials, S, hb, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                                 float(temperature), int(point_mass), seed, step, out_tokens, out_num_accepted, draws,
                                 device_status, cuda_stream)


def spec_shard_chunks(S, bounds) -> int:
    """Sums records per sequence and shard (chunks of the widest shard), 0 for invalid bounds."""
    hb = (ctypes.c_int32 * (S + 1))(*[int(v) for v in bounds])
    return lib.spec_shard_chunks(S, hb)


def spec_shard_sums(shard, S, bounds, shard_target, shard_draft, dtype, draws, seq_offsets, B, V, temperature, sums,
                    cuda_stream) -> int:
    """The draws' exact sums over one shard's slice, per chunk of SV_SHARD_CHUNK columns."""
    hb = (ctypes.c_int32 * (S + 1))(*[int(v) for v in bounds])
    return lib.spec_shard_sums(shard, S, hb, shard_target, shard_draft, dtype, draws, seq_offsets, B, V,
                               float(temperature), sums, cuda_stream)


def spec_shard_finish(shard, S, bounds, shard_target, shard_draft, dtype, draws, all_sums, seq_offsets, B, V,
                      temperature, out_tokens, cuda_stream) -> int:
    """The drawn tokens from the gathered sums (written by the owning shard, -1 elsewhere)."""
    hb = (ctypes.c_int32 * (S + 1))(*[int(v) for v in bounds])
    return lib.spec_shard_finish(shard, S, hb, shard_target, shard_draft, dtype, draws, all_sums, seq_offsets, B, V,
                                 float(temperature), out_tokens, cuda_stream)


def spec_verify_status_from_bits(bits: int) -> int:
    return lib.spec_verify_status_from_bits(bits)


def spec_verify_status_string(status: int) -> str:
    return lib.spec_verify_status_string(status).decode()


# ------------------------------------------------------------------------------------------------
# torch marshalling helpers
# ------------------------------------------------------------------------------------------------
def _ptr(t):
    return None if t is None else t.data_ptr()


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


class Call:
    """Device buffers of one verify call, allocated once and reused (workspace, outputs, status).

    ``run`` enqueues spec_verify_ex on the given stream and returns its host status code.
    """

    def __init__(self, B: int, V: int, max_gamma: int, R_t: int, R_d: int, device="cuda", debug=False):
        import torch
        self.B, self.V, self.max_gamma, self.R_t, self.R_d = B, V, max_gamma, R_t, R_d
        self.ws_bytes = spec_verify_workspace_size(B, V, max_gamma)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.out_tokens = torch.empty(R_t, dtype=torch.int32, device=device)
        self.out_n = torch.empty(B, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dbg = None
        self.dbg_struct = None
        if debug:
            self.dbg = dict(row_lse=torch.full((R_t + R_d,), float("nan"), dtype=torch.float64, device=device),
                            row_argmax=torch.full((R_t,), -7, dtype=torch.int32, device=device),
                            p_x=torch.full((R_d,), float("nan"), dtype=torch.float64, device=device),
                            q_x=torch.full((R_d,), float("nan"), dtype=torch.float64, device=device),
                            seq_mass=torch.full((B,), float("nan"), dtype=torch.float64, device=device),
                            beta=torch.full((R_d,), float("nan"), dtype=torch.float64, device=device))
            self.dbg_struct = SvDebug(*(self.dbg[k].data_ptr() for k in
                                        ("row_lse", "row_argmax", "p_x", "q_x", "seq_mass", "beta")), 0)

    def run(self, target, draft, draft_tokens, seq_offsets, gammas, temperature, seed, step, stream=None,
            clear_status=True, seq_base=0) -> int:
        import torch
        if clear_status:
            self.status.zero_()
        st = stream if stream is not None else torch.cuda.current_stream()
        return spec_verify_range(_ptr(target), _ptr(draft), dtype_code(target), _ptr(draft_tokens),
                                 _ptr(seq_offsets), _ptr(gammas), self.B, self.V, self.max_gamma, temperature,
                                 seed, step, seq_base, _ptr(self.out_tokens), _ptr(self.out_n), _ptr(self.status),
                                 _ptr(self.workspace), self.ws_bytes, self.dbg_struct, st.cuda_stream)

    def run_host(self, target, draft, draft_tokens, seq_offsets, gammas, temperature, seed, step, out_tokens,
                 out_num_accepted, staging, stream=None, clear_status=True) -> int:
        """Enqueue spec_verify_host: host tensors in (page-locked for asynchronous copies) and out, device
        staging tensors in ``staging`` (keys target, draft, draft_tokens, seq_offsets, gammas)."""
        import torch
        if clear_status:
            self.status.zero_()
        st = stream if stream is not None else torch.cuda.current_stream()
        dev = SvDeviceBuffers(_ptr(staging["target"]), _ptr(staging.get("draft")), _ptr(staging.get("draft_tokens")),
                              _ptr(staging["seq_offsets"]), _ptr(staging["gammas"]), _ptr(self.out_tokens),
                              _ptr(self.out_n))
        return spec_verify_host(_ptr(target), _ptr(draft), dtype_code(target), _ptr(draft_tokens), _ptr(seq_offsets),
                                _ptr(gammas), self.B, self.V, self.max_gamma, temperature, seed, step,
                                _ptr(out_tokens), _ptr(out_num_accepted), dev, _ptr(self.status),
                                _ptr(self.workspace), self.ws_bytes, st.cuda_stream)

    def commit(self, seq_offsets, history, capacity, lengths, next_tokens, stream=None) -> int:
        """Enqueue spec_verify_commit on this call's outputs (same stream, no host sync)."""
        import torch
        st = stream if stream is not None else torch.cuda.current_stream()
        return spec_verify_commit(_ptr(self.out_tokens), _ptr(self.out_n), _ptr(seq_offsets), self.B, _ptr(history),
                                  capacity, _ptr(lengths), _ptr(next_tokens), _ptr(self.status), st.cuda_stream)

    def run_fused(self, target, draft, draft_tokens, seq_offsets, gammas, temperature, seed, step, history,
                  capacity, lengths, next_tokens, stream=None, clear_status=True) -> int:
        """Enqueue spec_verify_fused (verify + post-verify update in one launch) on the given stream."""
        import torch
        if clear_status:
            self.status.zero_()
        st = stream if stream is not None else torch.cuda.current_stream()
        return spec_verify_fused(_ptr(target), _ptr(draft), dtype_code(target), _ptr(draft_tokens),
                                 _ptr(seq_offsets), _ptr(gammas), self.B, self.V, self.max_gamma, temperature,
                                 seed, step, _ptr(self.out_tokens), _ptr(self.out_n), _ptr(self.status),
                                 _ptr(self.workspace), self.ws_bytes, _ptr(history), capacity, _ptr(lengths),
                                 _ptr(next_tokens), st.cuda_stream)

    def status_bits(self) -> int:
        return int(self.status.item()) & 0xFFFFFFFF
