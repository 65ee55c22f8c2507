"""CPU oracle for the quantized paged KV cache path — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the GPU library computes,
written from the source pages (cited per function) and sharing no code with the
CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import it; the product package never does.

Modules
-------
formats     INT8 per-token-head codec (and with one scale per 32 values),
            E4M3 / E2M1 / NVFP4 codecs, BF16 rounding.
layout      reads the documented paged-pool layout (page, KV head, row).
attention   float64 decode attention, split ranges, log-sum-exp merge.
brute       pure-Python (math.fsum) attention for tiny inputs.
accounting  byte accounting of the formats (per token, per page, per pool).
rotation    the orthogonal rotation of K/V/q rows before quantization (Hadamard
            with a fixed sign vector), its fp32 butterfly arithmetic.

Parity status: every function here is pinned by the CPU tests under ``tests/``
(``test_oracle_*.py``) against closed forms printed on the pages, a library
routine that is independent of this code (torch's float8_e4m3fn cast, Python's
exact ``fractions`` arithmetic), brute force, or invariants.  No function here
is "parity unpinned".
"""
