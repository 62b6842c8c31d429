"""GB300-native sparse-MoE layer (route -> dispatch -> grouped SwiGLU experts with LoRA ->
combine) behind a C ABI (``include/moe.h``), with a thin ctypes binding in ``moe``."""
