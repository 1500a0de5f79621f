"""GB300-native (sm_103a) mixed-adapter batched LoRA delta.

The compute lives in liblora_delta.so (C ABI, include/lora_delta.h); the
``lora_delta`` module binds it.  ``workloads`` draws seeded synthetic inputs.
"""
