"""GB300-native paged MLA decode (placeholder; the binding is added with the library)."""
